// vt_rows.cu -- the row kernels: bf16 rows without penalties.
//
// The per-step decode sampler of the pages (TensorRT-LLM "Sampling": the
// temperature, min-p, top-k and top-p formulas; vllm.cpp pull request "the
// Gumbel draw that scanned 248,320 tokens on one thread": the seeded Gumbel
// draw over true global indices, lowest index on ties; Tenstorrent sampling
// README: log-softmax log-probs, one seed advance per sampled token), laid out
// for sm_103a as independent CTAs that never wait for one another:
//
//   pass kernel, one CTA per (row, slice of at most 76 KB):
//     * the slice arrives in shared memory by one bulk copy (mbarrier);
//     * pass A: the slice maximum (packed bf16 maxima per 16-byte vector,
//       kept per vector so later passes skip whole vectors), then the sum of
//       exponentials against it, the lowest-index argmax, and 8 group maxima
//       per thread;
//     * bf16 codes are exact bins: every element with one bf16 pattern has one
//       tempered value and one mass.  Rows whose kept set lies inside a small
//       top-k (and greedy rows' top-n) write the records of their elements
//       above a local lower bound of the k-th (n-th) largest value, taken from
//       the group maxima; rows whose kept set may reach far (top-p or min-p
//       without such a top-k) write a count per code slot below the slice
//       maximum; rows without a filter draw over every element;
//     * the partial results go to global memory, and the last CTA of the row
//       to arrive (one atomic per row) completes it: it merges the counts
//       (each CTA's slots shifted by its maximum's distance below the row's)
//       and walks them -- top-n boundary, min-p survivors, top-k boundary,
//       top-p over the top-k survivors renormalised, with masses summed in
//       exact fixed point -- then draws over the kept records and writes the
//       row, or leaves the walk for the draw kernel;
//   draw kernel, for the rows whose kept set needs every element: one CTA per
//     (row, slice) reads the slice again and scores its kept elements (a cheap
//     integer prefilter, then a certificate, skip nearly all of them); the
//     row's last CTA writes the token.
// Rows whose boundary falls where one slot holds several values (magnitudes
// below 2^-12, or the catch-all below the slot window), or whose records
// overflow, are handed to the selection kernel with their statistics.
#include "vt_device.cuh"
#include "vt_kernels.h"

#include <climits>

namespace vt {
namespace {

constexpr int kRT = 256;                 // threads per CTA of the row kernels
constexpr int kRW = kRT / 32;            // warps
constexpr int kSl = kRowSlots;           // code slots of the count histogram
constexpr int kSlCatch = kSl - 1;        // the last slot: everything below the window
constexpr int kSlPT = kSl / kRT;         // slots per thread in the walk
constexpr int kTinyE = 115;              // bf16 exponent field of 2^-12
constexpr int kGrp = 8;                  // group maxima per thread (thresholds)
constexpr int kPCap = 1024;              // top-k up to this: the records settle the row
constexpr int kListCap = 2048;           // boundary-slot indices one CTA can rank
constexpr int kSliceMax = 38912;         // elements per CTA at most (76 KB)
constexpr int kFinishRecCap = 5120;      // records the finish kernel holds (40 KB)
constexpr int kAllKept = -1;             // beta: every finite element is kept
constexpr int kNoKept = -2;              // beta: greedy row, no draw
constexpr int kThrAll = INT_MIN;         // threshold: every finite element
constexpr int kThrNone = INT_MAX;        // nothing written
static_assert(kSl % kRT == 0, "slots split evenly over the threads");
enum : int { kModeStats = 0, kModeRecords = 1, kModeCounts = 2, kModeAll = 3 };

// Signed code of a bf16 pattern, monotone in the value: magnitudes below
// 2^-12 and both zeros share code 0, every other value has a code of its own.
__device__ __forceinline__ int bcode(uint32_t u) {
  const int m = (int)(u & 0x7FFFu) - (kTinyE << 7) + 1;
  const int v = m > 0 ? m : 0;
  return (u & 0x8000u) ? -v : v;
}
// The bf16 value of a nonzero code.
__device__ __forceinline__ float bcode_value(int code) {
  const uint32_t mag = (uint32_t)((code < 0 ? -code : code) - 1 + (kTinyE << 7));
  return __uint_as_float(((code < 0 ? 0x8000u : 0u) | mag) << 16);
}
// The smallest value with code >= c (c = kThrAll: -inf).
__device__ __forceinline__ float code_floor_value(int c) {
  if (c == kThrAll) return -INFINITY;
  if (c == 0) return __uint_as_float(0xB97Fu << 16);  // -(2 - 2^-7) 2^-13
  return bcode_value(c);
}
// The largest magnitude code 0 stands for (an upper bound of |x|).
constexpr float kTinyMax = 0x1p-12f;

__device__ __forceinline__ void unpack8(const uint4& q, float* x) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint32_t bits8(const uint4& q, int i) {
  const uint32_t w = (i >> 1) == 0 ? q.x : (i >> 1) == 1 ? q.y : (i >> 1) == 2 ? q.z : q.w;
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}


// Records of candidate elements: code + 32768 in bits 52..36, 0xFFFFF - j in
// bits 35..16 and the bf16 pattern in bits 15..0, so that descending records
// are in the order (value descending, index ascending) wherever codes are
// single values, and the value is recovered exactly.
__device__ __forceinline__ uint64_t rec_make(int code, int j, uint32_t bits) {
  return ((uint64_t)(uint32_t)(code + 32768) << 36) | ((uint64_t)(0xFFFFFu - (uint32_t)j) << 16) |
         (uint64_t)bits;
}
__device__ __forceinline__ int rec_code(uint64_t r) { return (int)(r >> 36) - 32768; }
__device__ __forceinline__ int rec_j(uint64_t r) { return (int)(0xFFFFFu - ((uint32_t)(r >> 16) & 0xFFFFFu)); }
__device__ __forceinline__ float rec_x(uint64_t r) { return __uint_as_float(((uint32_t)r & 0xFFFFu) << 16); }

// The leader's walk over the merged slots, and what it found.
struct __align__(16) RRes {
  int action;              // 0: settled; 1: hand the row over
  int beta;                // kept boundary slot, kAllKept or kNoKept
  int qk;                  // kept elements of slot beta
  int sn;                  // top-n boundary slot (-1: no top-n)
  int cn;                  // top-n elements of slot sn
  int L3;                  // kept count
  float kth_z;             // tempered value of slot beta
  int pad;
};

struct __align__(16) RSmem {
  uint64_t full;           // bulk-copy completion
  RRes res;
  int flag, last, nrec, nlist, nlistn;
  unsigned int h256[256];  // threshold histogram
  float rf[4 * kRW];
  int ri[4 * kRW];
  unsigned long long ru[4 * kRW + 2];
  int bi[16];
  float bf[8];
  unsigned long long top[32];  // the row's top-n records
  int ntop;
  int delta[kRowMaxC];     // finisher: row slot = CTA r's slot + delta[r]
};

// ---------------------------------------------------------------------------
// block helpers (every thread of the CTA calls them)
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long w = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += w;
  }
  return v;
}

// Exclusive prefix over the CTA of one u64 per thread; *total = the sum.
__device__ unsigned long long rblock_excl(unsigned long long v, RSmem& s,
                                          unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long inc = warp_incl_u64(v, lane);
  if (lane == 31) s.ru[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long t = lane < kRW ? s.ru[lane] : 0ull;
    const unsigned long long ti = warp_incl_u64(t, lane);
    if (lane < kRW) s.ru[kRW + lane] = ti - t;
    if (lane == kRW - 1) s.ru[2 * kRW] = ti;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kRW + warp] + inc - v;
  *total = s.ru[2 * kRW];
  __syncthreads();
  return r;
}

__device__ int rblock_sum(int v, RSmem& s) {
  v = warp_sum_i(v);
  if ((threadIdx.x & 31) == 0) s.ri[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int t = threadIdx.x < kRW ? s.ri[threadIdx.x] : 0;
    t = warp_sum_i(t);
    if (threadIdx.x == 0) s.ri[kRW] = t;
  }
  __syncthreads();
  const int r = s.ri[kRW];
  __syncthreads();
  return r;
}

__device__ int rblock_max(int v, RSmem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) s.ri[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int t = threadIdx.x < kRW ? s.ri[threadIdx.x] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (threadIdx.x == 0) s.ri[kRW] = t;
  }
  __syncthreads();
  const int r = s.ri[kRW];
  __syncthreads();
  return r;
}

__device__ unsigned long long rblock_min_u64(unsigned long long v, RSmem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w < v ? w : v;
  }
  if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < kRW ? s.ru[threadIdx.x] : ~0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long w = __shfl_xor_sync(0xffffffffu, t, o);
      t = w < t ? w : t;
    }
    if (threadIdx.x == 0) s.ru[kRW] = t;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kRW];
  __syncthreads();
  return r;
}

// (score, index, payload) argmax over the CTA: larger score, then lower index.
__device__ void rblock_argmax(float& v, int& i, float& z, RSmem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    if (pair_better(v2, i2, v, i)) {
      v = v2;
      i = i2;
      z = z2;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    s.rf[warp] = v;
    s.ri[warp] = i;
    s.rf[kRW + warp] = z;
  }
  __syncthreads();
  if (warp == 0) {
    float tv = lane < kRW ? s.rf[lane] : -INFINITY;
    int ti = lane < kRW ? s.ri[lane] : INT_MAX;
    float tz = lane < kRW ? s.rf[kRW + lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, tv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ti, o);
      const float z2 = __shfl_xor_sync(0xffffffffu, tz, o);
      if (pair_better(v2, i2, tv, ti)) {
        tv = v2;
        ti = i2;
        tz = z2;
      }
    }
    if (lane == 0) {
      s.rf[2 * kRW] = tv;
      s.ri[2 * kRW] = ti;
      s.rf[2 * kRW + 1] = tz;
    }
  }
  __syncthreads();
  v = s.rf[2 * kRW];
  i = s.ri[2 * kRW];
  z = s.rf[2 * kRW + 1];
  __syncthreads();
}

// The c-th smallest (1-based) of n distinct values below 2^20 held in list[]
// (shared memory), by two rounds of 1024-bin counts in `bins` (shared, 1024
// words).  Every thread gets the result.
__device__ uint32_t rblock_kth_smallest(const uint32_t* list, int n, int c, uint32_t* bins,
                                        RSmem& s) {
  uint32_t prefix = 0;
  int want = c;
  for (int round = 0; round < 2; ++round) {
    const int shift = round == 0 ? 10 : 0;
    for (int b = threadIdx.x; b < 1024; b += kRT) bins[b] = 0u;
    __syncthreads();
    for (int e = threadIdx.x; e < n; e += kRT) {
      const uint32_t v = list[e];
      if (round == 0 || (v >> 10) == prefix) atomicAdd(&bins[(v >> shift) & 1023u], 1u);
    }
    __syncthreads();
    // 1024 bins over the threads: 2 each; find the bin holding the want-th
    constexpr int per = 1024 / kRT;
    unsigned long long mine = 0;
    for (int q = 0; q < per; ++q) mine += bins[threadIdx.x * per + q];
    unsigned long long tot;
    const unsigned long long ex = rblock_excl(mine, s, &tot);
    if (ex < (unsigned long long)want && ex + mine >= (unsigned long long)want) {
      unsigned long long run = ex;
      for (int q = 0; q < per; ++q) {
        const uint32_t cnt = bins[threadIdx.x * per + q];
        if (run + cnt >= (unsigned long long)want) {
          s.bi[0] = threadIdx.x * per + q;
          s.bi[1] = (int)run;
          break;
        }
        run += cnt;
      }
    }
    __syncthreads();
    const int bsel = s.bi[0];
    want -= s.bi[1];
    __syncthreads();
    prefix = round == 0 ? (uint32_t)bsel : ((prefix << 10) | (uint32_t)bsel);
  }
  return prefix;
}


// ---------------------------------------------------------------------------
// pass A: statistics of the slice (shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

struct Stats {
  float M;            // the slice maximum (every thread)
  float S;            // sum of exp(z_t - fl(M / T)) over the slice (every thread)
  int arg;            // lowest index of M (every thread; INT_MAX: none)
  bool bad;           // a NaN or +inf (every thread)
  float gm[kGrp];     // this thread's group maxima (vectors tid + k kRT, k = g mod kGrp)
};

// Two sweeps.  The first takes each 16-byte vector's maximum with packed bf16
// maxima (kept in vmax[v] as bf16 bits: later passes skip whole vectors), the
// thread's group maxima and its first vector holding its maximum; the slice
// maximum M and its lowest index follow.  The second sums
// 2^(z_t log2(e) - fl(M / T) log2(e)) with the reference product carried
// exactly as hi + lo: one FFMA (exact product, one rounding) and one add, so
// every exponent is the tempered difference to within an ulp at any scale.
// bf16 tempering fl(x / T) is strictly increasing in x (two bf16 values
// differ by at least 2^-8 relative, far above fp32 rounding), so the maximum
// and argmax of x are those of z_t.
__device__ Stats pass_stats(const uint4* sv, uint16_t* vmax, int nvec, int lo, float inv_t,
                            RSmem& s) {
  Stats o;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float rm = -INFINITY;
  int rv = -1;
#pragma unroll
  for (int g = 0; g < kGrp; ++g) o.gm[g] = -INFINITY;
  for (int v0 = tid; v0 < nvec; v0 += kGrp * kRT) {
#pragma unroll
    for (int g = 0; g < kGrp; ++g) {
      const int v = v0 + g * kRT;
      if (v < nvec) {
        const uint4 q = sv[v];
        const uint32_t m2 = bmax2(bmax2(q.x, q.y), bmax2(q.z, q.w));
        const float vm = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
        vmax[v] = (uint16_t)(__float_as_uint(vm) >> 16);
        o.gm[g] = fmaxf(o.gm[g], vm);
        if (vm > rm) {
          rm = vm;
          rv = v;
        }
      }
    }
  }
  // the slice maximum
  float m = warp_max(rm);
  if (lane == 0) s.rf[warp] = m;
  __syncthreads();
  if (warp == 0) {
    float t = lane < kRW ? s.rf[lane] : -INFINITY;
    t = warp_max(t);
    if (lane == 0) s.bf[0] = t;
  }
  __syncthreads();
  o.M = s.bf[0];
  // its lowest index: only threads whose maximum equals it hold one
  int j = INT_MAX;
  if (rv >= 0 && rm == o.M) {
    const uint4 q = sv[rv];
    float x[8];
    unpack8(q, x);
#pragma unroll
    for (int i = 7; i >= 0; --i)
      if (x[i] == o.M) j = lo + 8 * rv + i;
  }
  // the sum against fl(M / T)
  float rs = 0.f;
  bool nanf = false;
  if (o.M > -INFINITY) {
    const float Mt = __fmul_rn(o.M, inv_t);
    const float nh = __fmul_rn(-Mt, kLog2e);
    const float nl = __fmaf_rn(-Mt, kLog2e, -nh);
    // A vector whose tempered maximum is more than 30 below Mt adds less than
    // 8 e^-30 to a sum that is at least 1; over at most 2^20 elements the
    // skipped terms stay below 1e-7 of it.
    const float zcut = __fsub_rn(Mt, 30.0f);
    for (int v = tid; v < nvec; v += kRT) {
      if (__fmul_rn(__uint_as_float((uint32_t)vmax[v] << 16), inv_t) < zcut) continue;
      float x[8];
      unpack8(sv[v], x);
      float t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        t[i] = ex2_approx(__fadd_rn(__fmaf_rn(__fmul_rn(x[i], inv_t), kLog2e, nh), nl));
      rs += ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
    }
  } else {
    for (int v = tid; v < nvec; v += kRT) {
      float x[8];
      unpack8(sv[v], x);
#pragma unroll
      for (int i = 0; i < 8; ++i) nanf |= x[i] != x[i];
    }
  }
  nanf |= rs != rs;
  rs = warp_sum_f(rs);
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) j = min(j, __shfl_xor_sync(0xffffffffu, j, o2));
  const int anybad = __any_sync(0xffffffffu, nanf) ? 1 : 0;
  if (lane == 0) {
    s.rf[kRW + warp] = rs;
    s.ri[warp] = j;
    s.ri[kRW + warp] = anybad;
  }
  __syncthreads();
  if (warp == 0) {
    float t = lane < kRW ? s.rf[kRW + lane] : 0.f;
    int jj = lane < kRW ? s.ri[lane] : INT_MAX;
    int bb = lane < kRW ? s.ri[kRW + lane] : 0;
    t = warp_sum_f(t);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      jj = min(jj, __shfl_xor_sync(0xffffffffu, jj, o2));
      bb |= __shfl_xor_sync(0xffffffffu, bb, o2);
    }
    if (lane == 0) {
      s.bf[1] = t;
      s.bi[0] = jj;
      s.bi[1] = bb;
    }
  }
  __syncthreads();
  o.S = s.bf[1];
  o.arg = s.bi[0];
  o.bad = s.bi[1] != 0 || o.M == INFINITY;
  __syncthreads();
  return o;
}

// ---------------------------------------------------------------------------
// local thresholds: lower bounds of the slice's K-th largest element
// ---------------------------------------------------------------------------
// From the kGrp group maxima of every thread: at least K of the slice's
// elements are >= the K-th largest group maximum, so the slice's (and the
// row's) K-th largest element is >= it.  The bound is taken in bins of 16 codes
// below the CTA maximum's code (256 bins, the last one open), which only lowers
// it.  Returns codes (kThrAll: no bound) for Ka and Kb (0: not needed).
__device__ void local_thresholds(const float* gm, int cmax, int Ka, int Kb, RSmem& s, int* ta,
                                 int* tb) {
  for (int b = threadIdx.x; b < 256; b += kRT) s.h256[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int g = 0; g < kGrp; ++g) {
    if (gm[g] > -INFINITY) {
      const int d = cmax - bcode(__float_as_uint(gm[g]) >> 16);
      if (d >= 0) atomicAdd(&s.h256[d >= 255 * 16 ? 255 : (d >> 4)], 1u);
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t cnt[8], tot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      cnt[q] = s.h256[8 * lane + q];
      tot += cnt[q];
    }
    uint32_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t w = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += w;
    }
    const uint32_t before = inc - tot;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t K = (uint32_t)(which == 0 ? Ka : Kb);
      if (lane == 0) s.bi[4 + which] = kThrAll;
      __syncwarp();
      if (K > 0 && before < K && inc >= K) {
        uint32_t run = before;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run < K && run + cnt[q] >= K) {
            const int b = 8 * lane + q;
            s.bi[4 + which] = b == 255 ? kThrAll : cmax - 16 * b - 15;
          }
          run += cnt[q];
        }
      }
      __syncwarp();
    }
  }
  __syncthreads();
  *ta = Ka > 0 ? s.bi[4] : kThrAll;
  *tb = Kb > 0 ? s.bi[5] : kThrAll;
  __syncthreads();
}

// The smallest code whose largest value passes min-p against the tempered
// maximum m_t (a lower bound of the survivors' codes: the row maximum is at
// least m_t).  A 32-way search by one warp (every lane gets the result);
// monotone because min-p is.
__device__ int minp_code_warp(float inv_t, float m_t, double lmp, int cmax) {
  const int lane = threadIdx.x & 31;
  auto pass = [&](int c) {
    const float v = c == 0 ? kTinyMax : bcode_value(c);
    return minp_pass(__fmul_rn(v, inv_t), m_t, lmp);
  };
  int lo = -bcode(0x7F80u), hi = cmax;  // lo: the code of -inf (never passes); hi passes
  while (hi - lo > 1) {
    const int span = hi - lo;
    const int step = (span + 31) / 32;
    const int c = min(hi, lo + (lane + 1) * step);
    const unsigned ok = __ballot_sync(0xffffffffu, pass(c));
    const int first = __ffs(ok) - 1;  // hi passes, so some lane with c == hi passes
    const int chi = min(hi, lo + (first + 1) * step);
    lo = first == 0 ? lo : min(hi, lo + first * step);
    hi = chi;
  }
  return hi;
}

// ---------------------------------------------------------------------------
// pass H: counts per code slot below the CTA maximum
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned int pass_counts(const uint4* sv, const uint16_t* vmax,
                                                    int nvec, float tau_x, int cmax,
                                                    uint32_t* hist) {
  unsigned int catch_cnt = 0;
  for (int v = threadIdx.x; v < nvec; v += kRT) {
    if (!(__uint_as_float((uint32_t)vmax[v] << 16) >= tau_x)) continue;  // nothing counted
    const uint4 q = sv[v];
    float x[8];
    unpack8(q, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (x[i] >= tau_x && x[i] > -INFINITY) {
        const int sl = cmax - bcode(bits8(q, i));
        if (sl < kSlCatch) atomicAdd(&hist[sl], 1u);
        else ++catch_cnt;
      }
    }
  }
  return catch_cnt;
}


// ---------------------------------------------------------------------------
// the walk over the merged code slots
// ---------------------------------------------------------------------------
struct WalkIn {
  int n;                    // top-n
  bool greedy, topk, topp, minp;
  bool need_cut;            // the counts cover the kept set only if top-k cuts inside them
  int top_k;
  float top_p;
  double lmp;
  float inv_t, m_t;
  int cmax;                 // code of the row maximum
  int Smax;                 // row slots [0, Smax] hold every element of their value
  bool full;                // every finite element is counted (the catch-all too)
  unsigned int catch_row;   // counted elements below the window
};

// Row slot S stands for the bf16 value of code cmax - S (slot 0: the row
// maximum).  Its elements share one tempered value, so its count settles the
// filters and count x mass its share of any sum.  Two slots are not single
// values: the code-0 slot (|x| < 2^-12) and the catch-all (everything below
// the window); their masses are carried as [low, high] bounds, and a
// boundary that falls in them, or a decision the bounds leave open, hands the
// row over.  cnt[S] holds the row's count of slot S for S <= Smax.  Writes
// s.res.  Every thread of the CTA calls it.
__device__ __noinline__ void walk_slots(const WalkIn& w, const uint32_t* hist, RSmem& s) {
  const int tid = threadIdx.x;
  const int S0 = tid * kSlPT;
  if (tid == 0) {
    s.flag = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) s.bi[i] = -1;
  }
  uint32_t cnt[kSlPT];
#pragma unroll
  for (int q = 0; q < kSlPT; ++q) cnt[q] = (S0 + q <= w.Smax) ? hist[S0 + q] : 0u;
  __syncthreads();  // s.bi initialised

  const float m_t = w.m_t;
  auto slot_z = [&](int S) { return __fmul_rn(bcode_value(w.cmax - S), w.inv_t); };
  const float z_tlo = __fmul_rn(-kTinyMax, w.inv_t), z_thi = __fmul_rn(kTinyMax, w.inv_t);
  const int code_bot = w.cmax - kSlCatch;  // the largest code of the catch-all
  const float z_bot = __fmul_rn(code_bot == 0 ? kTinyMax : bcode_value(code_bot), w.inv_t);

  // ---- survivors of min-p, per slot ----
  uint32_t cs[kSlPT];
  unsigned int ta = 0, ts = 0;
#pragma unroll
  for (int q = 0; q < kSlPT; ++q) {
    const int S = S0 + q;
    bool sv = true;
    if (w.minp && cnt[q] != 0u) {
      if (w.cmax - S == 0) {
        const bool plo = minp_pass(z_tlo, m_t, w.lmp), phi = minp_pass(z_thi, m_t, w.lmp);
        sv = plo;
        if (phi && !plo) atomicOr(&s.flag, 1);
      } else {
        sv = minp_pass(slot_z(S), m_t, w.lmp);
      }
    }
    cs[q] = sv ? cnt[q] : 0u;
    ta += cnt[q];
    ts += cs[q];
  }
  unsigned long long TA, TS;
  const unsigned long long ea = rblock_excl(ta, s, &TA);
  const unsigned long long es = rblock_excl(ts, s, &TS);
  unsigned long long catch_surv = 0;
  if (w.full && w.catch_row > 0u) {
    if (w.minp) {
      if (minp_pass(z_bot, m_t, w.lmp) && tid == 0) atomicOr(&s.flag, 1);
    } else {
      catch_surv = w.catch_row;
    }
  }

  // ---- top-n boundary (all elements) and top-k boundary (survivors) ----
  auto find_count = [&](unsigned long long before, const uint32_t* c, unsigned long long mine,
                        unsigned long long K, int out) {
    if (before < K && before + mine >= K) {
      unsigned long long run = before;
#pragma unroll
      for (int q = 0; q < kSlPT; ++q) {
        if (run < K && run + c[q] >= K) {
          const int S = S0 + q;
          if (w.cmax - S == 0) atomicOr(&s.flag, 1);
          s.bi[out] = S;
          s.bi[out + 1] = (int)(K - run);
        }
        run += c[q];
      }
    }
  };
  if (w.n > 0) {
    if (TA < (unsigned long long)w.n) {
      if (tid == 0) atomicOr(&s.flag, 1);  // the top-n reaches past the counted slots
    } else {
      find_count(ea, cnt, ta, (unsigned long long)w.n, 0);
    }
  }
  bool cut = false;
  if (w.topk) {
    const unsigned long long K = (unsigned long long)w.top_k;
    if (K <= TS) {
      cut = true;
      find_count(es, cs, ts, K, 2);
    } else if (K <= TS + catch_surv || w.need_cut) {
      if (tid == 0) atomicOr(&s.flag, 1);  // the top-k boundary past the counted slots
    }
  }
  __syncthreads();
  const int sn = w.n > 0 ? s.bi[0] : -1, cn_tot = s.bi[1];
  const int sk = s.bi[2], ck = s.bi[3];
  __syncthreads();

  auto c_eff = [&](int q) -> uint32_t {
    const int S = S0 + q;
    if (!cut) return cs[q];
    return S < sk ? cs[q] : (S == sk ? (uint32_t)ck : 0u);
  };

  // ---- the kept boundary ----
  int beta = kAllKept, qk = 0;
  if (w.greedy) {
    beta = kNoKept;
  } else if (w.topp) {
    const unsigned long long mu_tlo = mass_fixed(z_tlo, m_t), mu_thi = mass_fixed(z_thi, m_t);
    unsigned long long tlo = 0, thi = 0;
#pragma unroll
    for (int q = 0; q < kSlPT; ++q) {
      const uint32_t ce = c_eff(q);
      if (ce == 0u) continue;
      const int S = S0 + q;
      if (w.cmax - S == 0) {
        tlo += ce * mu_tlo;
        thi += ce * mu_thi;
      } else {
        const unsigned long long m = ce * mass_fixed(slot_z(S), m_t);
        tlo += m;
        thi += m;
      }
    }
    unsigned long long Wlo, Whi;
    const unsigned long long Alo = rblock_excl(tlo, s, &Wlo);
    const unsigned long long Ahi = rblock_excl(thi, s, &Whi);
    if (!cut) Whi += catch_surv * mass_fixed(z_bot, m_t);
    const double p = (double)w.top_p;
    const unsigned long long Tlo = (unsigned long long)((double)Wlo * p);
    const unsigned long long Thi = (unsigned long long)((double)Whi * p);
    // the last kept element: exclusive prefix <= T; searched at both ends of
    // the bounds (the most and the least inclusive reading)
#pragma unroll
    for (int var = 0; var < 2; ++var) {
      const unsigned long long A0 = var == 0 ? Alo : Ahi;
      const unsigned long long mine = var == 0 ? tlo : thi;
      const unsigned long long T = var == 0 ? Thi : Tlo;
      if (A0 <= T && A0 + mine > T) {
        unsigned long long run = A0;
        bool done = false;
#pragma unroll
        for (int q = 0; q < kSlPT; ++q) {
          const uint32_t ce = c_eff(q);
          if (done || ce == 0u) continue;
          const int S = S0 + q;
          const bool tiny = w.cmax - S == 0;
          const unsigned long long mu =
              tiny ? (var == 0 ? mu_tlo : mu_thi) : mass_fixed(slot_z(S), m_t);
          const unsigned long long mm = ce * mu;
          if (run + mm > T) {
            if (tiny) atomicOr(&s.flag, 1);
            unsigned long long kq = (T - run) / mu + 1ull;
            if (kq > ce) kq = ce;
            s.bi[6 + 2 * var] = S;
            s.bi[7 + 2 * var] = (int)kq;
            done = true;
          }
          run += mm;
        }
      }
    }
    __syncthreads();
    if (tid == 0 && (s.bi[6] < 0 || s.bi[6] != s.bi[8] || s.bi[7] != s.bi[9]))
      atomicOr(&s.flag, 1);  // past the counted slots, or left open by the bounds
    __syncthreads();
    beta = s.bi[6];
    qk = s.bi[7];
  } else if (cut) {
    beta = sk;
    qk = ck;
  } else if (w.minp) {
    int last = -1;
#pragma unroll
    for (int q = 0; q < kSlPT; ++q)
      if (cs[q] != 0u) last = S0 + q;
    beta = rblock_max(last, s);
    if (beta >= 0 && beta >= S0 && beta < S0 + kSlPT) s.bi[10] = (int)cs[beta - S0];
    __syncthreads();
    qk = s.bi[10];
  }
  // kept count: survivors before beta plus the kept ones of beta
  if (beta >= 0 && beta >= S0 && beta < S0 + kSlPT) {
    unsigned long long run = es;
#pragma unroll
    for (int q = 0; q < kSlPT; ++q)
      if (S0 + q < beta) run += cs[q];
    s.bi[11] = (int)(run + (unsigned long long)qk);
  }
  __syncthreads();
  if (tid == 0) {
    RRes& R = s.res;
    if (beta >= 0 && qk < 1) s.flag |= 1;
    R.beta = beta;
    R.qk = qk;
    R.sn = sn;
    R.cn = cn_tot;
    R.L3 = beta >= 0 ? s.bi[11] : (beta == kNoKept ? 1 : 0);
    R.kth_z = beta >= 0 ? slot_z(beta) : 0.f;
    R.action = s.flag ? 1 : 0;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// shared pieces of the two kernels
// ---------------------------------------------------------------------------
// Row parameters as the kernels use them.
struct RowCfg {
  bool greedy, topk, topp, minp;
  int top_k, n, mode;
  float inv_t, top_p;
  double lmp;
};
__device__ __forceinline__ RowCfg row_cfg(const RowArgs& a, int row, const RowParams& P) {
  RowCfg c;
  c.greedy = (P.flags & kRowGreedy) != 0;
  c.inv_t = P.inv_t;
  c.top_p = P.top_p;
  bool topp = (P.flags & kRowTopP) != 0;
  if (P.flags & kRowDecay) {  // the decayed top_p; 1 (the start) filters nothing
    c.top_p = a.decay[row].p;
    topp = c.top_p < 1.0f;
  }
  c.topp = topp && !c.greedy;
  c.top_k = P.top_k;
  c.topk = !c.greedy && P.top_k > 1 && P.top_k < a.V;
  c.minp = !c.greedy && (P.flags & kRowMinP) != 0;
  c.lmp = P.log_min_p;
  c.n = a.n_logprobs;
  if (c.greedy) c.mode = c.n > 0 ? kModeRecords : kModeStats;
  else if (!c.topk && !c.topp && !c.minp) c.mode = kModeAll;
  else if (c.topk && c.top_k <= kPCap) c.mode = kModeRecords;
  else c.mode = kModeCounts;
  return c;
}

// Copy CTA `rank`'s slice of `row` into shared memory: one bulk copy of its
// whole 16-byte units (aligned rows), plain loads for the rest; -inf past the
// end up to whole vectors.  Returns false when the bounded wait ran out.
__device__ bool load_slice(const RowArgs& a, int row, int lo, int nel, int nvec, uint8_t* buf,
                           RSmem& s) {
  const uint16_t* src = reinterpret_cast<const uint16_t*>(a.logits) + (int64_t)row * a.ld + lo;
  const uint32_t bulk = a.aligned ? (((uint32_t)nel * 2u) & ~15u) : 0u;
  if (threadIdx.x == 0 && bulk) {
    mbar_init(&s.full, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&s.full, bulk);
    bulk_copy_g2s(buf, src, bulk, &s.full);
  }
  uint16_t* e16 = reinterpret_cast<uint16_t*>(buf);
  for (int k = (int)(bulk >> 1) + threadIdx.x; k < nel; k += kRT) e16[k] = src[k];
  for (int k = nel + threadIdx.x; k < 8 * nvec; k += kRT) e16[k] = 0xFF80u;
  __syncthreads();  // the mbarrier initialised, the plain part stored
  bool ok = true;
  if (bulk) ok = mbar_wait_bounded(&s.full, 0u);
  return ok;
}

// The best Gumbel score over elements offered one at a time: a 24-bit
// integer prefilter, then the certificate, then the exact score.  An element
// beats the best bs only if -ln u < e^(z - bs) <= e^(zmax - bs) = E, and
// -ln u >= 1 - u, so only if u > 1 - E: b >= blo (a 2^-8 margin and one unit
// cover the fp32 rounding).
struct Draw {
  float bs = -INFINITY, bz = 0.f;
  int bj = INT_MAX;
  uint32_t blo = 0u;
  float zmax;
  __device__ explicit Draw(float zmax_) : zmax(zmax_) {}
  // The noise bound for elements whose tempered value is at most z.
  __device__ __forceinline__ uint32_t bound(float z) const {
    if (bs == -INFINITY) return 0u;
    const float E = ex2_approx(__fmul_rn(__fsub_rn(z, bs), kLog2e)) * 1.00390625f;
    const float th = (1.0f - E) * 16777216.0f;
    return (E < 1.0f && th > 1.0f) ? (uint32_t)th - 1u : 0u;
  }
  __device__ __forceinline__ void offer(float z, int j, uint32_t bits) {
    if (bits < blo) return;
    if (!may_beat(z, bs, bits)) return;
    const float sc = gumbel_score(z, bits);
    if (pair_better(sc, j, bs, bj)) {
      bs = sc;
      bj = j;
      bz = z;
      const float E = ex2_approx(__fmul_rn(__fsub_rn(zmax, bs), kLog2e)) * 1.00390625f;
      const float th = (1.0f - E) * 16777216.0f;
      blo = (E < 1.0f && th > 1.0f) ? (uint32_t)th - 1u : 0u;
    }
  }
};

// Outputs of a row without a token: -1, NaN log-probs, the status; the seed
// still advances.  All threads of one CTA call it.
__device__ void write_bad(const RowArgs& a, int row, int status, int err) {
  const int n = a.n_logprobs;
  if ((int)threadIdx.x < n) {
    a.out_topk_ids[(int64_t)row * n + threadIdx.x] = -1;
    a.out_topk_logprobs[(int64_t)row * n + threadIdx.x] = __int_as_float(0x7fc00000);
  }
  if (threadIdx.x == 0) {
    a.out_tokens[row] = -1;
    if (a.out_logprobs) a.out_logprobs[row] = __int_as_float(0x7fc00000);
    a.row_status[row] = status;
    a.dbg_kth_value[row] = __int_as_float(0x7fc00000);
    a.dbg_kth_index[row] = -1;
    a.dbg_kept[row] = 0;
    a.seeds[row] += kSeedStep;
    if (err) atomicOr(a.err_word, err);
  }
}

// The token and its row data.  One thread calls it.
__device__ void write_token(const RowArgs& a, int row, const RowParams& P, int tok, float ztok,
                            float m_t, float lnS, float kz, int kj, int L3, int err) {
  a.out_tokens[row] = tok;
  if (a.out_logprobs) a.out_logprobs[row] = (ztok - m_t) - lnS;
  a.row_status[row] = kRowOk;
  a.dbg_kth_value[row] = kz;
  a.dbg_kth_index[row] = kj;
  a.dbg_kept[row] = L3;
  a.seeds[row] += kSeedStep;
  if (P.flags & kRowDecay) {  // [TensorRT-LLM "Sampling", top-p decay]
    DecayState& d = a.decay[row];
    const float qd = __fmul_rn(d.p, d.decay);
    d.p = tok == d.reset_id ? P.top_p : (qd < d.p_min ? d.p_min : qd);
  }
  if (err) atomicOr(a.err_word, err);
}

// Hand a row to the selection kernel with its statistics.  One thread.
__device__ void hand_over(const RowArgs& a, int row, float m_t, float lnS, float xmax, int arg,
                          int err) {
  SlowRow sr;
  sr.m_t = m_t;
  sr.lnS = lnS;
  sr.xmax = xmax;
  sr.bi_topn = (uint32_t)arg | (a.n_logprobs == 0 ? 0x80000000u : 0u);
  a.slow[row] = sr;
  a.slow_list[atomicAdd(a.slow_ctl, 1u)] = row;
  if (err) atomicOr(a.err_word, err);
}

// ---------------------------------------------------------------------------
// the pass kernel: one CTA per (row, slice); the row's last CTA completes it
// ---------------------------------------------------------------------------
__device__ void finish_row(const RowArgs& a, int row, const RowParams& P, const RowCfg& c,
                           uint8_t* buf, uint32_t* hist, uint32_t* list, RSmem& s);

__global__ void __launch_bounds__(kRT, 2) row_pass_kernel(const RowArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ RSmem s;
  const int tid = threadIdx.x;
  const int C = a.C;
  const int q = (int)blockIdx.x / C, rank = (int)blockIdx.x % C;
  if (q >= a.norder) return;
  const int row = a.order[q];
  if (row >= a.B) return;
  const int lo = rank * a.slice;
  const int nel = max(0, min(lo + a.slice, a.V) - lo);
  const int nvec = (nel + 7) >> 3;
  uint8_t* buf = dsm;
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + a.buf_bytes);
  uint16_t* vmax = reinterpret_cast<uint16_t*>(hist + kSl);
  unsigned long long* tr = a.trace ? a.trace + ((size_t)row * C + rank) * kTraceSlots : nullptr;
#define VT_RTRACE(k)                                 \
  do {                                               \
    if (tr && tid == 0) tr[(k)] = global_timer_ns(); \
  } while (0)
  VT_RTRACE(0);
  int err = load_slice(a, row, lo, nel, nvec, buf, s) ? 0 : kErrTimeout;
  VT_RTRACE(1);
  const uint4* sv = reinterpret_cast<const uint4*>(buf);
  const RowParams P = a.params[row];
  const RowCfg c = row_cfg(a, row, P);

  // ---- pass A ----
  const Stats st = pass_stats(sv, vmax, nvec, lo, c.inv_t, s);
  const int cmax = st.M > -INFINITY ? bcode(__float_as_uint(st.M) >> 16) : -bcode(0x7F80u);
  const float Mt = st.M > -INFINITY ? __fmul_rn(st.M, c.inv_t) : -INFINITY;
  VT_RTRACE(2);

  // ---- records, counts, or the draw over every element ----
  int thr = kThrNone, thr_n = kThrNone, nrec = 0, fin = 0;
  unsigned int catch_cnt = 0u;
  unsigned long long lastk = ~0ull;
  Draw d(Mt);
  if (c.mode != kModeStats && !st.bad) {
    int tn = kThrAll, tk = kThrAll;
    const int Kk = (c.mode == kModeRecords && c.topk && c.top_k <= kGrp * kRT) ? c.top_k : 0;
    local_thresholds(st.gm, cmax, c.n, Kk, s, &tn, &tk);
    if (c.mode == kModeRecords) {
      if (c.greedy) {
        thr = tn;
      } else {
        int tkept = Kk > 0 ? tk : kThrAll;
        if (c.minp) {
          if ((tid >> 5) == 0) {
            const int mc = Mt > -INFINITY ? minp_code_warp(c.inv_t, Mt, c.lmp, cmax) : kThrAll;
            if ((tid & 31) == 0) s.bi[6] = mc;
          }
          __syncthreads();
          tkept = max(tkept, s.bi[6]);
          __syncthreads();
        }
        thr = c.n > 0 ? min(tn, tkept) : tkept;
      }
      thr_n = thr;
    } else {
      thr_n = c.n > 0 ? tn : kThrNone;
    }
    // records of the elements with code >= the record threshold
    const int rthr = c.mode == kModeRecords ? thr : thr_n;
    if (rthr != kThrNone) {
      const float tx = code_floor_value(rthr);
      if (tid == 0) s.nrec = 0;
      __syncthreads();
      uint64_t* out = a.cand + ((size_t)row * C + rank) * a.cand_cap;
      const int lane = tid & 31;
      for (int v0 = tid - lane; v0 < nvec; v0 += kRT) {  // warp-uniform trip count
        const int v = v0 + lane;
        uint32_t m = 0u;
        uint4 qv = make_uint4(0u, 0u, 0u, 0u);
        if (v < nvec && __uint_as_float((uint32_t)vmax[v] << 16) >= tx) {
          qv = sv[v];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x = __uint_as_float(bits8(qv, i) << 16);
            m |= (uint32_t)(x >= tx && x > -INFINITY) << i;
          }
        }
        if (!__any_sync(0xffffffffu, m != 0u)) continue;
        // one shared atomic per warp: each lane's records at its prefix
        const int cnt = __popc(m);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const int wtot = __shfl_sync(0xffffffffu, incl, 31);
        int base = 0;
        if (lane == 31 && wtot > 0) base = atomicAdd(&s.nrec, wtot);
        base = __shfl_sync(0xffffffffu, base, 31);
        int pos = base + incl - cnt;
        while (m) {
          const int i = __ffs(m) - 1;
          m &= m - 1u;
          const uint32_t bits = bits8(qv, i);
          if (pos < a.cand_cap) out[pos] = rec_make(bcode(bits), lo + 8 * v + i, bits);
          ++pos;
        }
      }
      __syncthreads();
      nrec = s.nrec;
    }
    if (c.mode == kModeCounts) {  // a count per code slot below the slice maximum
      thr = kThrAll;
      uint4* h4 = reinterpret_cast<uint4*>(hist);
      for (int k = tid; k < kSl / 4; k += kRT) h4[k] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      catch_cnt =
          (unsigned int)rblock_sum((int)pass_counts(sv, vmax, nvec, -INFINITY, cmax, hist), s);
      uint4* g4 = reinterpret_cast<uint4*>(a.ghist + ((size_t)row * C + rank) * kSl);
      for (int k = tid; k < kSl / 4; k += kRT) g4[k] = h4[k];
    } else if (c.mode == kModeAll) {  // no filter: every finite element is kept
      const uint64_t key = row_key(a.seeds[row], row);
      for (int v = tid; v < nvec; v += kRT) {
        const uint4 qv = sv[v];
        float x[8];
        unpack8(qv, x);
        uint64_t h[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) h[w] = pair_hash(key, lo + 8 * v + 2 * w);
#pragma unroll
        for (int q2 = 0; q2 < 8; ++q2) {
          if (x[q2] > -INFINITY) {
            const int j = lo + 8 * v + q2;
            const float z = __fmul_rn(x[q2], c.inv_t);
            d.offer(z, j, (q2 & 1) ? bits_odd(h[q2 >> 1]) : bits_even(h[q2 >> 1]));
            const unsigned long long k = elem_key(z, (uint32_t)j);
            lastk = k < lastk ? k : lastk;
            ++fin;
          }
        }
      }
      rblock_argmax(d.bs, d.bj, d.bz, s);
      lastk = rblock_min_u64(lastk, s);
      fin = rblock_sum(fin, s);
    }
  }
  VT_RTRACE(3);
  if (tid == 0) {
    RowPartG& pt = a.part[(size_t)row * C + rank];
    pt.xmax = st.M;
    pt.s = st.S;
    pt.arg = st.arg;
    pt.bad = st.bad ? 1 : 0;
    pt.cmax = cmax;
    pt.thr = thr;
    pt.thr_n = thr_n;
    pt.catch_cnt = catch_cnt;
    pt.ncand = nrec;
    pt.err = err;
    pt.best_s = d.bs;
    pt.best_z = d.bz;
    pt.best_j = d.bj;
    pt.kth_j = -1;
    pt.last_key = lastk;
    pt.fin = fin;
  }
#undef VT_RTRACE
}

// ---------------------------------------------------------------------------
// the finish kernel: one CTA per row, after the pass kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRT, 3) row_finish_kernel(const RowArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ RSmem s;
  const int q = (int)blockIdx.x;
  if (q >= a.norder) return;
  const int row = a.order[q];
  if (row >= a.B) return;
  unsigned long long* tr = a.trace ? a.trace + (size_t)row * a.C * kTraceSlots : nullptr;
  if (tr && threadIdx.x == 0) tr[4] = global_timer_ns();
  const RowParams P = a.params[row];
  const RowCfg c = row_cfg(a, row, P);
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm);
  uint32_t* list = hist + kSl;
  uint8_t* recbuf = reinterpret_cast<uint8_t*>(list + kListCap);
  finish_row(a, row, P, c, recbuf, hist, list, s);
  if (tr && threadIdx.x == 0) tr[5] = global_timer_ns();
}

// The top-n from records whose slot < sn (all) or == sn (the first cn by
// index), ordered (value descending, index ascending) by their exact values.
__device__ void write_topn(const RowArgs& a, int row, const RowCfg& c, const uint64_t* recs,
                           int nrec, int cmax_row, int sn, int cn, int nsn, float m_t, float lnS,
                           uint32_t* list, uint32_t* bins, RSmem& s, int* err) {
  const int tid = threadIdx.x;
  const int code_n = cmax_row - sn;
  if (tid == 0) {
    s.ntop = 0;
    s.nlistn = 0;
  }
  __syncthreads();
  const bool all_sn = cn == nsn;
  for (int e = tid; e < nrec; e += kRT) {
    const uint64_t r = recs[e];
    const int code = rec_code(r);
    if (code > code_n || (code == code_n && all_sn)) {
      const int pos = atomicAdd(&s.ntop, 1);
      if (pos < 32) s.top[pos] = r;
    } else if (code == code_n) {
      const int pos = atomicAdd(&s.nlistn, 1);
      if (pos < kListCap) list[pos] = (uint32_t)rec_j(r);
    }
  }
  __syncthreads();
  if (!all_sn) {
    const int nl = min(s.nlistn, kListCap);
    const uint32_t kth = rblock_kth_smallest(list, nl, cn, bins, s);
    for (int e = tid; e < nrec; e += kRT) {
      const uint64_t r = recs[e];
      if (rec_code(r) == code_n && (uint32_t)rec_j(r) <= kth) {
        const int pos = atomicAdd(&s.ntop, 1);
        if (pos < 32) s.top[pos] = r;
      }
    }
    __syncthreads();
  }
  const int n = c.n;
  if (tid < 32) {
    const int g = min(s.ntop, 32);
    unsigned long long k = 0ull;
    float z = 0.f;
    int j = -1;
    if (tid < g) {
      const uint64_t r = s.top[tid];
      j = rec_j(r);
      z = __fmul_rn(rec_x(r), c.inv_t);
      k = elem_key(z, (uint32_t)j);
    }
    int rk = 0;
    for (int t = 0; t < g; ++t) rk += __shfl_sync(0xffffffffu, k, t) > k;
    if (tid < g && rk < n) {
      a.out_topk_ids[(int64_t)row * n + rk] = j;
      a.out_topk_logprobs[(int64_t)row * n + rk] = (z - m_t) - lnS;
    }
    if (tid == 0 && g != n) *err |= kErrInternal;
  }
  __syncthreads();
}

__device__ void finish_row(const RowArgs& a, int row, const RowParams& P, const RowCfg& c,
                           uint8_t* buf, uint32_t* hist, uint32_t* list, RSmem& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = a.C;
  const RowPartG* parts = a.part + (size_t)row * C;
  // ---- the row's statistics from every CTA's partials ----
  if (warp == 0) {
    float xm = -INFINITY, mt = -INFINITY, sm = 0.f, bs = -INFINITY, bz = 0.f;
    int arg = INT_MAX, bd = 0, th = INT_MIN, thn = INT_MIN, er = 0, cm = INT_MIN, ovf = 0;
    int bj = INT_MAX, fn = 0;
    unsigned int ct = 0u;
    unsigned long long lk = ~0ull;
    if (lane < C) {
      const RowPartG* pp = parts + lane;
      xm = __ldcg(&pp->xmax);
      mt = xm > -INFINITY ? __fmul_rn(xm, c.inv_t) : -INFINITY;
      sm = __ldcg(&pp->s);
      arg = __ldcg(&pp->arg);
      bd = __ldcg(&pp->bad);
      th = __ldcg(&pp->thr);
      thn = __ldcg(&pp->thr_n);
      ct = __ldcg(&pp->catch_cnt);
      ovf = __ldcg(&pp->ncand) > a.cand_cap;
      er = __ldcg(&pp->err);
      cm = __ldcg(&pp->cmax);
      bs = __ldcg(&pp->best_s);
      bz = __ldcg(&pp->best_z);
      bj = __ldcg(&pp->best_j);
      lk = __ldcg(&pp->last_key);
      fn = __ldcg(&pp->fin);
    }
    const int my_cmax = cm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float x2 = __shfl_xor_sync(0xffffffffu, xm, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, arg, o);
      const float mt2 = __shfl_xor_sync(0xffffffffu, mt, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
      if (pair_better(x2, a2, xm, arg)) {
        xm = x2;
        arg = a2;
      }
      lse_combine(mt, sm, mt2, s2, kLog2e);
      const float b2 = __shfl_xor_sync(0xffffffffu, bs, o);
      const int j2 = __shfl_xor_sync(0xffffffffu, bj, o);
      const float z2 = __shfl_xor_sync(0xffffffffu, bz, o);
      if (pair_better(b2, j2, bs, bj)) {
        bs = b2;
        bj = j2;
        bz = z2;
      }
      const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, lk, o);
      lk = l2 < lk ? l2 : lk;
      bd |= __shfl_xor_sync(0xffffffffu, bd, o);
      er |= __shfl_xor_sync(0xffffffffu, er, o);
      ovf |= __shfl_xor_sync(0xffffffffu, ovf, o);
      th = max(th, __shfl_xor_sync(0xffffffffu, th, o));
      thn = max(thn, __shfl_xor_sync(0xffffffffu, thn, o));
      cm = max(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      ct += __shfl_xor_sync(0xffffffffu, ct, o);
      fn += __shfl_xor_sync(0xffffffffu, fn, o);
    }
    if (lane < C) s.delta[lane] = cm - my_cmax;
    if (lane == 0) {
      s.bf[0] = xm;
      s.bf[1] = mt;
      s.bf[2] = sm;
      s.bf[3] = bz;
      s.bi[0] = arg;
      s.bi[1] = bd || xm == INFINITY;
      s.bi[2] = th;
      s.bi[3] = thn;
      s.bi[4] = (int)ct;
      s.bi[5] = er;
      s.bi[6] = cm;
      s.bi[7] = ovf;
      s.bi[8] = bj;
      s.bi[9] = fn;
      s.ru[0] = lk;
    }
  }
  __syncthreads();
  const float xmax = s.bf[0], m_t = s.bf[1], S = s.bf[2], bz = s.bf[3];
  const int arg = s.bi[0], bad = s.bi[1], thr = s.bi[2], thrn = s.bi[3];
  const unsigned int catch_tot = (unsigned int)s.bi[4];
  int err = s.bi[5];
  const int cmax = s.bi[6], ovf = s.bi[7], bj = s.bi[8], fn = s.bi[9];
  const unsigned long long lk = s.ru[0];
  const float lnS = logf(S);
  __syncthreads();
  auto done = [&]() {};
  if (bad || xmax == -INFINITY) {
    write_bad(a, row, bad ? kRowNonfinite : kRowEmpty, err);
    done();
    return;
  }
  if (c.mode == kModeStats) {  // greedy, no top-n
    if (tid == 0) write_token(a, row, P, arg, m_t, m_t, lnS, m_t, arg, 1, err);
    done();
    return;
  }
  if (c.mode == kModeAll && c.n == 0) {
    if (tid == 0) write_token(a, row, P, bj, bz, m_t, lnS, key_z(lk), (int)key_idx(lk), fn, err);
    done();
    return;
  }

  // ---- the records this row needs, in shared memory ----
  uint64_t* recs = reinterpret_cast<uint64_t*>(buf);
  const int rcap = kFinishRecCap;
  const int rthr = c.mode == kModeRecords ? thr : thrn;
  int nrec = 0;
  if (rthr != kThrNone) {
    if (tid == 0) s.nrec = 0;
    __syncthreads();
    if (!ovf) {
      // every CTA's record count, then all records in one flat sweep
      int* ncum = s.ri;  // [C + 1] exclusive prefix of the counts
      if (tid < 32) {
        int v = tid < C ? __ldcg(&parts[tid].ncand) : 0;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, inc, o);
          if (tid >= o) inc += t;
        }
        if (tid == 0) ncum[0] = 0;
        if (tid < C) ncum[tid + 1] = inc;
      }
      __syncthreads();
      const int total = ncum[C];
      const uint64_t* base = a.cand + (size_t)row * C * a.cand_cap;
      for (int e0 = tid; e0 < total; e0 += 4 * kRT) {
        uint64_t rec[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = e0 + u * kRT;
          rec[u] = ~0ull;
          if (e < total) {
            int r = 0;
            while (r + 1 < C && e >= ncum[r + 1]) ++r;
            rec[u] = __ldcg(base + (size_t)r * a.cand_cap + (e - ncum[r]));
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (rec[u] != ~0ull && rec_code(rec[u]) >= rthr) {
            const int pos = atomicAdd(&s.nrec, 1);
            if (pos < rcap) recs[pos] = rec[u];
          }
        }
      }
    }
    __syncthreads();
    nrec = s.nrec;
  }
  if (ovf || nrec > rcap) {
    if (tid == 0) hand_over(a, row, m_t, lnS, xmax, arg, err);
    done();
    return;
  }

  // ---- counts per row slot ----
  WalkIn w;
  w.n = c.n;
  w.greedy = c.greedy || c.mode == kModeAll;
  w.topk = c.topk && !w.greedy;
  w.topp = c.topp && !w.greedy;
  w.minp = c.minp && !w.greedy;
  w.need_cut = c.mode == kModeRecords && w.topk && !w.minp;
  w.top_k = c.top_k;
  w.top_p = c.top_p;
  w.lmp = c.lmp;
  w.inv_t = c.inv_t;
  w.m_t = m_t;
  w.cmax = cmax;
  if (c.mode == kModeCounts) {
    // every CTA's counts, shifted by its maximum's distance below the row's
    unsigned int extra = 0u;
    uint32_t cnt[kSlPT];
#pragma unroll
    for (int q = 0; q < kSlPT; ++q) cnt[q] = 0u;
    const int S0 = tid * kSlPT;
    for (int r = 0; r < C; ++r) {
      const uint32_t* gh = a.ghist + ((size_t)row * C + r) * kSl;
      const int d = s.delta[r];
      uint32_t v[kSlPT];
#pragma unroll
      for (int q = 0; q < kSlPT; ++q) {
        const int sl = S0 + q - d;
        v[q] = (S0 + q < kSlCatch && sl >= 0) ? __ldcg(gh + sl) : 0u;
      }
#pragma unroll
      for (int q = 0; q < kSlPT; ++q) cnt[q] += v[q];
      for (int sl = max(kSlCatch - d, 0) + tid; sl < kSlCatch; sl += kRT) extra += __ldcg(gh + sl);
    }
#pragma unroll
    for (int q = 0; q < kSlPT; ++q) hist[S0 + q] = cnt[q];
    w.catch_row = catch_tot + (unsigned int)rblock_sum((int)extra, s);
    w.Smax = kSlCatch - 1;
    w.full = true;
  } else {
    uint4* h4 = reinterpret_cast<uint4*>(hist);
    for (int k = tid; k < kSl / 4; k += kRT) h4[k] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    int beyond = 0;
    for (int e = tid; e < nrec; e += kRT) {
      const int sl = cmax - rec_code(recs[e]);
      if (sl < kSlCatch) atomicAdd(&hist[sl], 1u);
      else ++beyond;
    }
    w.catch_row = (unsigned int)rblock_sum(beyond, s);
    const long long Sstar = rthr == kThrAll ? (long long)INT_MAX : (long long)cmax - rthr;
    w.full = Sstar >= kSlCatch;
    w.Smax = (int)(Sstar < kSlCatch - 1 ? Sstar : kSlCatch - 1);
  }
  __syncthreads();
  walk_slots(w, hist, s);
  const RRes R = s.res;
  // counts the later steps need, before the histogram is reused as scratch
  const int nsn = R.sn >= 0 ? (int)hist[R.sn] : 0;
  const int nbeta = R.beta >= 0 ? (int)hist[R.beta] : 0;
  __syncthreads();
  bool give = R.action != 0;
  if (R.sn >= 0 && R.cn < nsn && nsn > kListCap) give = true;
  if (c.mode == kModeRecords && R.beta >= 0 && R.qk < nbeta && nbeta > kListCap) give = true;
  if (give) {
    if (tid == 0) hand_over(a, row, m_t, lnS, xmax, arg, err);
    done();
    return;
  }
  if (c.n > 0) write_topn(a, row, c, recs, nrec, cmax, R.sn, R.cn, nsn, m_t, lnS, list, hist, s, &err);

  if (c.mode == kModeCounts) {
    // the draw kernel finishes the row: each CTA's share of the boundary slot
    if (tid < C) {
      const int d = s.delta[tid];
      const int sl = R.beta - d;
      s.ri[tid] = (sl >= 0 && sl < kSlCatch) ? (int)__ldcg(a.ghist + ((size_t)row * C + tid) * kSl + sl) : 0;
    }
    __syncthreads();
    if (tid == 0) {
      RowWalk W;
      W.action = 0;
      W.beta = R.beta;
      W.L3 = R.L3;
      W.kth_z = R.kth_z;
      W.m_t = m_t;
      W.lnS = lnS;
      W.cmax = cmax;
      W.last_rank = -1;
      int pre = 0;
      bool ok = R.beta >= 0;
      for (int r = 0; r < C; ++r) {
        const int nb = s.ri[r];
        const int cb = min(max(R.qk - pre, 0), nb);
        if (pre < R.qk && R.qk <= pre + nb) W.last_rank = r;
        if (cb > 0 && cb < nb && nb > kListCap) ok = false;
        W.cb[r] = cb;
        W.nb[r] = nb;
        pre += nb;
      }
      if (W.last_rank < 0) ok = false;
      if (!ok) {
        hand_over(a, row, m_t, lnS, xmax, arg, err);
      } else {
        a.walk[row] = W;
        __threadfence();
        a.flist[atomicAdd(&a.fctl[0], 1u)] = row;
        if (err) atomicOr(a.err_word, err);
      }
    }
    done();
    return;
  }
  if (c.mode == kModeAll || c.greedy) {
    if (tid == 0) {
      if (c.greedy) write_token(a, row, P, arg, m_t, m_t, lnS, m_t, arg, 1, err);
      else write_token(a, row, P, bj, bz, m_t, lnS, key_z(lk), (int)key_idx(lk), fn, err);
    }
    done();
    return;
  }

  // ---- records: the draw over the kept set ----
  const int code_b = cmax - R.beta;
  const bool all_b = R.qk == nbeta;
  const uint64_t key = row_key(a.seeds[row], row);
  Draw dr(m_t);
  int kthj = -1;
  if (tid == 0) s.nlist = 0;
  __syncthreads();
  for (int e = tid; e < nrec; e += kRT) {
    const uint64_t r = recs[e];
    const int code = rec_code(r);
    const int j = rec_j(r);
    if (code > code_b || (code == code_b && all_b)) {
      dr.offer(__fmul_rn(rec_x(r), c.inv_t), j, noise_bits(key, j));
      if (code == code_b) kthj = max(kthj, j);
    } else if (code == code_b) {
      const int pos = atomicAdd(&s.nlist, 1);
      if (pos < kListCap) list[pos] = (uint32_t)j;
    }
  }
  __syncthreads();
  if (!all_b) {
    const uint32_t kth = rblock_kth_smallest(list, min(s.nlist, kListCap), R.qk, hist, s);
    for (int e = tid; e < nrec; e += kRT) {
      const uint64_t r = recs[e];
      const int j = rec_j(r);
      if (rec_code(r) == code_b && (uint32_t)j <= kth)
        dr.offer(__fmul_rn(rec_x(r), c.inv_t), j, noise_bits(key, j));
    }
    kthj = (int)kth;
  }
  rblock_argmax(dr.bs, dr.bj, dr.bz, s);
  kthj = rblock_max(kthj, s);
  if (tid == 0) {
    if (dr.bj == INT_MAX || kthj < 0) err |= kErrInternal;
    write_token(a, row, P, dr.bj, dr.bz, m_t, lnS, R.kth_z, kthj, R.L3, err);
  }
  done();
}

// ---------------------------------------------------------------------------
// the draw kernel: rows whose kept set needs every element
// ---------------------------------------------------------------------------
// One CTA per (listed row, slice).  Elements above the boundary value x_b are
// kept, and of those equal to it the first cb (by index) of this CTA; the
// row's last CTA combines the best scores and writes the token.  The grid's
// last CTA clears the list for the next call.
__global__ void __launch_bounds__(kRT, 2) row_draw_kernel(const RowArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ RSmem s;
  const int tid = threadIdx.x;
  const int C = a.C;
  const int i = (int)blockIdx.x / C, rank = (int)blockIdx.x % C;
  const int nf = (int)__ldcg(&a.fctl[0]);
  if (i < nf) {
    const int row = __ldcg(&a.flist[i]);
    const RowWalk* wp = a.walk + row;
    const int beta = __ldcg(&wp->beta), L3 = __ldcg(&wp->L3), cmax = __ldcg(&wp->cmax);
    const int cb = __ldcg(&wp->cb[rank]), nb = __ldcg(&wp->nb[rank]);
    const int last_rank = __ldcg(&wp->last_rank);
    const float m_t = __ldcg(&wp->m_t), lnS = __ldcg(&wp->lnS), kth_z = __ldcg(&wp->kth_z);
    const int lo = rank * a.slice;
    const int nel = max(0, min(lo + a.slice, a.V) - lo);
    const int nvec = (nel + 7) >> 3;
    uint8_t* buf = dsm;
    uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + a.buf_bytes);
    uint32_t* list = hist + kSl;
    unsigned long long* tr = a.trace ? a.trace + ((size_t)row * C + rank) * kTraceSlots : nullptr;
    if (tr && tid == 0) tr[6] = global_timer_ns();
    int err = load_slice(a, row, lo, nel, nvec, buf, s) ? 0 : kErrTimeout;
    if (tr && tid == 0) tr[7] = global_timer_ns();
    const RowParams P = a.params[row];
    const float inv_t = P.inv_t;
    const uint4* sv = reinterpret_cast<const uint4*>(buf);
    const float xb = bcode_value(cmax - beta);
    const bool all_b = cb == nb;
    const uint64_t key = row_key(a.seeds[row], row);
    Draw d(m_t);
    int kthj = -1;
    if (tid == 0) s.nlist = 0;
    __syncthreads();
    for (int v = tid; v < nvec; v += kRT) {
      const uint4 qv = sv[v];
      const uint32_t m2 = bmax2(bmax2(qv.x, qv.y), bmax2(qv.z, qv.w));
      if (!(fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u)) >= xb)) continue;
      float x[8];
      unpack8(qv, x);
      uint32_t km = 0u, eq = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        km |= (uint32_t)(x[q] > xb) << q;
        eq |= (uint32_t)(x[q] == xb) << q;
      }
      while (eq) {  // elements of the boundary slot (few)
        const int q = __ffs(eq) - 1;
        eq &= eq - 1u;
        const int j = lo + 8 * v + q;
        if (all_b) {
          km |= 1u << q;
          kthj = max(kthj, j);
        } else if (cb > 0) {
          const int pos = atomicAdd(&s.nlist, 1);
          if (pos < kListCap) list[pos] = (uint32_t)j;
        }
      }
      if (km) {
        // the vector's four hashes together (independent chains overlap); an
        // element can beat the best only if its noise clears the bound the
        // vector's own maximum sets (one ex2 per vector, one compare each)
        uint64_t h[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) h[w] = pair_hash(key, lo + 8 * v + 2 * w);
        const float zv = __fmul_rn(fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u)), inv_t);
        const uint32_t bv = d.bound(zv);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t bits = (q & 1) ? bits_odd(h[q >> 1]) : bits_even(h[q >> 1]);
          if ((km & (1u << q)) && bits >= bv) d.offer(__fmul_rn(x[q], inv_t), lo + 8 * v + q, bits);
        }
      }
    }
    __syncthreads();
    if (!all_b && cb > 0) {
      const int nl = min(s.nlist, kListCap);
      if (s.nlist != nb && tid == 0) err |= kErrInternal;
      const uint32_t kth = rblock_kth_smallest(list, nl, cb, hist, s);
      const uint16_t* e16 = reinterpret_cast<const uint16_t*>(buf);
      for (int e = tid; e < nl; e += kRT) {
        const int j = (int)list[e];
        if ((uint32_t)j <= kth)
          d.offer(__fmul_rn(__uint_as_float((uint32_t)e16[j - lo] << 16), inv_t), j,
                  noise_bits(key, j));
      }
      kthj = (int)kth;
    }
    if (tr && tid == 0) tr[8] = global_timer_ns();
    rblock_argmax(d.bs, d.bj, d.bz, s);
    kthj = rblock_max(kthj, s);
    if (tid == 0) {
      RowPartG& pt = a.part[(size_t)row * C + rank];
      pt.best_s = d.bs;
      pt.best_j = d.bj;
      pt.best_z = d.bz;
      pt.kth_j = rank == last_rank ? kthj : -1;
      pt.err = err;
      __threadfence();
      s.last = atomicAdd(&a.ctl[row], 1u) == (unsigned int)(C - 1);
    }
    __syncthreads();
    if (s.last && tid == 0) {
      __threadfence();
      float bs = -INFINITY, bz = 0.f;
      int bj = INT_MAX, kj = -1, er = 0;
      for (int r = 0; r < C; ++r) {
        const RowPartG* pp = a.part + (size_t)row * C + r;
        const float b2 = __ldcg(&pp->best_s);
        const int j2 = __ldcg(&pp->best_j);
        if (pair_better(b2, j2, bs, bj)) {
          bs = b2;
          bj = j2;
          bz = __ldcg(&pp->best_z);
        }
        if (r == last_rank) kj = __ldcg(&pp->kth_j);
        er |= __ldcg(&pp->err);
      }
      if (bj == INT_MAX || kj < 0) er |= kErrInternal;
      write_token(a, row, P, bj, bz, m_t, lnS, kth_z, kj, L3, er);
      a.ctl[row] = 0u;
      if (tr) tr[9] = global_timer_ns();
    }
  }
  // the grid's last CTA clears the list for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&a.fctl[1], 1u) == gridDim.x - 1) {
      a.fctl[2] = a.fctl[0];
      a.fctl[0] = 0u;
      a.fctl[1] = 0u;
      __threadfence();
    }
  }
}

}  // namespace
}  // namespace vt

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace vt {

constexpr size_t kFinishSmem = (size_t)kSl * 4 + (size_t)kListCap * 4 + (size_t)kFinishRecCap * 8;

RowPlan plan_rows(int B, int V) {
  (void)B;
  RowPlan p{};
  const int C = (V + kSliceMax - 1) / kSliceMax;
  if (V < 1 || C > kRowMaxC) return p;
  int slice = (V + C - 1) / C;
  slice = (slice + 7) & ~7;
  const uint32_t buf = (uint32_t)(((size_t)slice * 2 + 127) & ~(size_t)127);
  const size_t vbytes = (((size_t)slice / 8 * 2 + 15) & ~(size_t)15);
  const size_t smem = buf + (size_t)kSl * 4 + (vbytes > (size_t)kListCap * 4 ? vbytes : (size_t)kListCap * 4);
  if (cudaFuncSetAttribute(row_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(row_draw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return p;
  }
  if (cudaFuncSetAttribute(row_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kFinishSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return p;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_pass_kernel, kRT, smem) !=
          cudaSuccess ||
      per_sm < 1) {
    (void)cudaGetLastError();
    return p;
  }
  p.cluster = C;
  p.slice = slice;
  p.buf_bytes = buf;
  p.smem = smem;
  p.clusters = per_sm;
  return p;
}

cudaError_t launch_rows(const RowArgs& args, const RowPlan& plan, int draw_rows,
                        cudaStream_t stream) {
  if (plan.cluster < 1 || args.norder < 1) return cudaErrorInvalidConfiguration;
  row_pass_kernel<<<(unsigned)(args.norder * plan.cluster), kRT, plan.smem, stream>>>(args);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  row_finish_kernel<<<(unsigned)args.norder, kRT, kFinishSmem, stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess || draw_rows < 1) return e;
  row_draw_kernel<<<(unsigned)(draw_rows * plan.cluster), kRT, plan.smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace vt
