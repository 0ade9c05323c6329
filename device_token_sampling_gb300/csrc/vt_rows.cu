// vt_rows.cu -- the persistent row kernel: bf16 rows without penalties.
//
// The per-step decode sampler of the pages (TensorRT-LLM "Sampling": the
// temperature, min-p, top-k and top-p formulas; vllm.cpp pull request "the
// Gumbel draw that scanned 248,320 tokens on one thread": the seeded Gumbel
// draw over true global indices, lowest index on ties; Tenstorrent sampling
// README: log-softmax log-probs, one seed advance per sampled token), laid out
// for sm_103a so that HBM streams each logit once while every later pass reads
// shared memory:
//
//   * persistent thread-block clusters of C CTAs loop over the rows (heaviest
//     first, in a host-made order); CTA r of a cluster owns elements
//     [r * slice, (r + 1) * slice) of each of its rows;
//   * each CTA holds its slice of the current row in one shared-memory
//     buffer while one bulk copy fills the other with the slice of the
//     cluster's next row (double buffering, one mbarrier per buffer);
//   * pass A (statistics): row maximum, sum of exponentials, lowest-index
//     argmax, and four group maxima per thread;
//   * pass H (counts): bf16 codes are exact bins -- every element with one
//     bf16 pattern has the same tempered value and the same mass -- so a count
//     per code slot below the CTA's own maximum settles min-p, top-k, top-p
//     and the top-n exactly.  Rows whose kept set is small count only the
//     elements above a local lower bound of their k-th (n-th) largest value,
//     taken from the group maxima; top-p rows count every element;
//   * barrier 1; the leader CTA merges the C histograms (each shifted by the
//     distance of its CTA's maximum below the row's) and walks the slots:
//     top-n boundary, min-p survivors, top-k boundary, top-p over the top-k
//     survivors renormalised, with masses summed in exact fixed point;
//   * barrier 2; pass D draws over the kept elements (Gumbel scores, with a
//     cheap certificate that skips elements that cannot win) and sends the
//     top-n to the leader; the kept elements of the boundary slot are the
//     lowest-indexed ones, selected per CTA;
//   * barrier 3; the leader writes the row's outputs.
// Rows whose boundary falls where one slot holds several values (the slot of
// magnitudes below 2^-12, or the catch-all below the slot window) are handed
// to the selection kernel with their statistics, exactly as the streaming
// kernel hands rows over.
#include "vt_device.cuh"
#include "vt_kernels.h"

#include <climits>

namespace cg = cooperative_groups;

namespace vt {
namespace {

constexpr int kRT = 512;                 // threads per CTA of the row kernel
constexpr int kRW = kRT / 32;            // warps
constexpr int kSl = 4096;                // code slots of the count histogram
constexpr int kSlCatch = kSl - 1;        // the last slot: everything below the window
constexpr int kSlPT = kSl / kRT;         // slots per thread in the walk
constexpr int kTinyE = 115;              // bf16 exponent field of 2^-12
constexpr int kGrp = 4;                  // group maxima per thread (thresholds)
constexpr int kListCap = 2048;           // boundary-slot indices one CTA can rank
constexpr int kGatherCap = 64;           // top-n keys the leader gathers
constexpr int kRMaxC = 16;               // CTAs per cluster at most
constexpr int kAllKept = -1;             // beta: every finite element is kept
constexpr int kNoKept = -2;              // beta: greedy row, no draw
constexpr int kThrAll = INT_MIN;         // histogram threshold: every finite element
constexpr int kThrNone = INT_MAX;        // no histogram
static_assert(kSl % kRT == 0, "slots split evenly over the threads");

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

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// What a CTA publishes for the row (read by the others over DSMEM).
struct __align__(16) RPart {
  float xmax;              // CTA maximum before temperature (-inf: none)
  float s;                 // sum of exp(z_t - fl(xmax / T)) over the slice
  int arg;                 // lowest index of xmax (INT_MAX: none)
  int bad;                 // a NaN or +inf
  int cmax;                // code of xmax
  int thr;                 // the histogram counted finite elements with code >= thr
  unsigned int catch_cnt;  // counted elements below the CTA's slot window
  int err;
  // after the draw pass
  float best_s, best_z;    // best Gumbel score and its tempered value
  int best_j;
  int kth_j;               // the row's last kept index when this CTA holds it (-1)
  unsigned long long last_key;  // rows keeping everything: the order's last element here
  int fin;                 // rows keeping everything: finite elements here
  int pad0;
};

// The leader's walk, read by every CTA after barrier 2.
struct __align__(16) RRes {
  int action;              // 0: draw and gather; 1: handed to the selection kernel
  int beta;                // kept boundary slot, kAllKept or kNoKept
  int sn;                  // top-n boundary slot (-1: no top-n)
  int L3;                  // kept count
  float kth_z;             // tempered value of the last kept element (slot rows)
  int last_rank;           // CTA holding the last kept element of slot beta
  int cb[kRMaxC];          // kept elements of slot beta per CTA
  int nb[kRMaxC];          // elements of slot beta per CTA
  int cn[kRMaxC];          // top-n elements of slot sn per CTA
  int nn[kRMaxC];          // elements of slot sn per CTA
};

struct __align__(16) RSmem {
  uint64_t full[2];        // bulk-copy completion, one per slice buffer
  RPart part[2];           // by row parity
  RRes res;                // leader: this row's walk
  RRes rl;                 // every CTA: the leader's walk
  uint64_t gather[kGatherCap];  // leader: top-n keys
  int gcount;
  int nlist, nlistn;       // boundary-slot indices listed by this CTA
  int flag;
  unsigned int h256[256];  // threshold histogram
  float rf[4 * kRW];
  int ri[4 * kRW];
  unsigned long long ru[4 * kRW + 2];
  int bi[16];
  float bf[8];
  unsigned long long bu[8];
  int delta[kRMaxC];       // row slot = CTA r's slot + delta[r]
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
struct Stats {
  float rm, rmt, rs;   // thread maximum, its tempered value, sum of exp(z_t - rmt)
  int j;               // lowest index of rm among this thread's elements (INT_MAX: none)
  bool bad;            // a NaN seen (a +inf shows as rm)
  float gm[kGrp];      // maxima of the thread's vectors k = 0, 1, 2, 3 (mod 4)
};

// One pass over the thread's 16-byte vectors v = tid + k * kRT: the running
// maximum rm with the sum rs of exp(z_t - fl(rm / T)), rescaled when rm grows;
// the first vector holding rm; a NaN flag; and each vector's maximum into
// vmax[v] (bf16 bits), which lets the later passes skip whole vectors.  Each
// term is 2^(z_t log2(e) - fl(rm / T) log2(e)) with the reference product
// carried exactly as hi + lo: one FFMA (exact product, one rounding) and one
// add, so the exponent is the tempered difference to within an ulp at any
// scale.  bf16 tempering fl(x / T) is strictly increasing in x (two bf16
// values differ by at least 2^-8 relative, far above fp32 rounding), so the
// maximum and argmax of x are those of z_t.
__device__ __forceinline__ Stats pass_stats(const uint4* sv, uint16_t* vmax, int nvec, int lo,
                                            float inv_t) {
  Stats o;
  o.rm = -INFINITY;
  o.rmt = -INFINITY;
  o.rs = 0.f;
  o.j = INT_MAX;
  o.bad = false;
#pragma unroll
  for (int g = 0; g < kGrp; ++g) o.gm[g] = -INFINITY;
  float nb_hi = 0.f, nb_lo = 0.f;  // -fl(rm / T) log2(e) = nb_hi + nb_lo
  int rv = -1;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kGrp * kRT) {
#pragma unroll
    for (int g = 0; g < kGrp; ++g) {
      const int v = v0 + g * kRT;
      if (v < nvec) {
        float x[8];
        unpack8(sv[v], x);
        const float vm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                               fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
        vmax[v] = (uint16_t)(__float_as_uint(vm) >> 16);
        o.gm[g] = fmaxf(o.gm[g], vm);
        if (vm > o.rm) {
          const float vmt = __fmul_rn(vm, inv_t);
          const float nh = __fmul_rn(-vmt, kLog2e);
          const float nl = __fmaf_rn(-vmt, kLog2e, -nh);
          o.rs = (o.rm == -INFINITY)
                     ? 0.f
                     : o.rs * ex2_approx(__fadd_rn(__fmaf_rn(o.rmt, kLog2e, nh), nl));
          o.rm = vm;
          o.rmt = vmt;
          nb_hi = nh;
          nb_lo = nl;
          rv = v;
        }
        if (o.rm > -INFINITY) {
          float t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            t[i] = ex2_approx(__fadd_rn(__fmaf_rn(__fmul_rn(x[i], inv_t), kLog2e, nb_hi), nb_lo));
          o.rs += ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) o.bad |= x[i] != x[i];
        }
      }
    }
  }
  o.bad |= o.rs != o.rs;
  if (rv >= 0) {
    float x[8];
    unpack8(sv[rv], x);
    int first = 7;
#pragma unroll
    for (int i = 7; i >= 0; --i)
      if (x[i] == o.rm) first = i;
    o.j = lo + 8 * rv + first;
  }
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
// the leader's walk over the merged code slots
// ---------------------------------------------------------------------------
struct WalkIn {
  int C;
  int n;                    // top-n
  bool greedy, topk, topp, minp;
  int top_k;
  float top_p;
  double lmp;
  float inv_t, m_t;
  int cmax;                 // code of the row maximum
  int Smax;                 // row slots [0, Smax] hold every element of their value
  bool full;                // every CTA counted every finite element
  unsigned int catch_tot;   // the CTAs' own catch-all counts
  int delta[kRMaxC];        // row slot = CTA r's slot + delta[r]
};

// Row slot S stands for the bf16 value of code cmax - S (slot 0: the row
// maximum).  Its elements share one tempered value, so its count settles the
// filters and count x mass its share of any sum.  Two slots are not single
// values: the code-0 slot (|x| < 2^-12) and the catch-all (everything below
// the window); their masses are carried as [low, high] bounds, and a
// boundary that falls in them, or a decision the bounds leave open, hands the
// row over.  Writes s.res.  Every thread of the leader CTA calls it.
__device__ __noinline__ void leader_walk(const WalkIn& w, uint32_t* hist, RSmem& s) {
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const int S0 = tid * kSlPT;
  if (tid == 0) {
    s.flag = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) s.bi[i] = -1;
  }
  // ---- merge: row slot S of CTA r is its slot S - delta[r] ----
  uint32_t cnt[kSlPT];
#pragma unroll
  for (int q = 0; q < kSlPT; ++q) cnt[q] = 0u;
  unsigned int extra = 0;
  for (int r = 0; r < w.C; ++r) {
    const uint32_t* hr = cluster.map_shared_rank(hist, r);
    const int d = w.delta[r];
#pragma unroll
    for (int q = 0; q < kSlPT; ++q) {
      const int S = S0 + q, sl = S - d;
      if (S <= w.Smax && sl >= 0) cnt[q] += hr[sl];
    }
    // slots of CTA r that fall below the row's window join the catch-all
    if (w.full)
      for (int sl = max(kSlCatch - d, 0) + tid; sl < kSlCatch; sl += kRT) extra += hr[sl];
  }
  const unsigned int catch_row = w.full ? w.catch_tot + (unsigned int)rblock_sum((int)extra, s) : 0u;
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
  if (w.full && catch_row > 0u) {
    if (w.minp) {
      if (minp_pass(z_bot, m_t, w.lmp) && tid == 0) atomicOr(&s.flag, 1);
    } else {
      catch_surv = catch_row;
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
      if (tid == 0) atomicOr(&s.flag, 1);  // the top-n reaches past the window
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
    } else if (K <= TS + catch_surv) {
      if (tid == 0) atomicOr(&s.flag, 1);  // the top-k boundary in the catch-all
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
      atomicOr(&s.flag, 1);  // past the window, or left open by the bounds
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

  // ---- per-CTA shares of the two boundary slots ----
  if (tid < w.C) {
    const uint32_t* hr = cluster.map_shared_rank(hist, tid);
    const int d = w.delta[tid];
    s.res.nb[tid] = (beta >= 0 && beta - d >= 0) ? (int)hr[beta - d] : 0;
    s.res.nn[tid] = (sn >= 0 && sn - d >= 0) ? (int)hr[sn - d] : 0;
  }
  __syncthreads();
  if (tid == 0) {
    RRes& R = s.res;
    int pre = 0, pren = 0, sum_b = 0;
    R.last_rank = -1;
    for (int r = 0; r < w.C; ++r) {
      const int nb = R.nb[r], nn = R.nn[r];
      const int cb = beta >= 0 ? min(max(qk - pre, 0), nb) : 0;
      const int cn = sn >= 0 ? min(max(cn_tot - pren, 0), nn) : 0;
      if (beta >= 0 && pre < qk && qk <= pre + nb) R.last_rank = r;
      if ((cb > 0 && cb < nb && nb > kListCap) || (cn > 0 && cn < nn && nn > kListCap)) s.flag |= 1;
      R.cb[r] = cb;
      R.cn[r] = cn;
      pre += nb;
      pren += nn;
      sum_b += nb;
    }
    if (beta >= 0 && (R.last_rank < 0 || qk < 1)) s.flag |= 1;
    R.beta = beta;
    R.sn = sn;
    R.L3 = beta >= 0 ? s.bi[11] : (beta == kNoKept ? 1 : 0);
    R.kth_z = beta >= 0 ? slot_z(beta) : 0.f;
    R.action = s.flag ? 1 : 0;
  }
  __syncthreads();
}


// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRT, 1) rows_kernel(const RowArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ RSmem s;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int cid = (int)blockIdx.x / C, ncl = (int)gridDim.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool leader = rank == 0;
  const int lo = rank * a.slice;
  const int hi = min(lo + a.slice, a.V);
  const int nel = max(0, hi - lo);
  const int nvec = (nel + 7) >> 3;
  const int n = a.n_logprobs;
  auto buf_at = [&](int bf) { return dsm + (size_t)bf * a.buf_bytes; };
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + 2 * (size_t)a.buf_bytes);
  uint32_t* list_b = hist + kSl;
  uint32_t* list_n = list_b + kListCap;
  uint16_t* vmax = reinterpret_cast<uint16_t*>(list_n + kListCap);  // [nvec] vector maxima
  // aligned rows: one bulk copy of the slice's whole 16-byte units, the last
  // (< 8) elements by plain loads; other rows: plain loads of the whole slice
  const uint32_t bulk = a.aligned ? (((uint32_t)nel * 2u) & ~15u) : 0u;
  const int tail0 = a.aligned ? (int)(bulk >> 1) : 0;
  const int ntail = a.aligned ? nel - tail0 : 0;
  auto row_src = [&](int row) {
    return reinterpret_cast<const uint16_t*>(a.logits) + (int64_t)row * a.ld + lo;
  };
  auto next_q = [&](int q) {
    while (q < a.norder && a.order[q] >= a.B) q += ncl;
    return q;
  };

  // -inf past the slice's end up to whole vectors (never written again)
  for (int bf = 0; bf < 2; ++bf) {
    uint16_t* e = reinterpret_cast<uint16_t*>(buf_at(bf));
    for (int k = nel + tid; k < 8 * nvec; k += kRT) e[k] = 0xFF80u;
  }
  if (tid == 0) {
    mbar_init(&s.full[0], 1);
    mbar_init(&s.full[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int row, int bf) {  // thread 0
    if (bulk) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&s.full[bf], bulk);
      bulk_copy_g2s(buf_at(bf), row_src(row), bulk, &s.full[bf]);
    }
  };
  int q = next_q(cid);
  if (q < a.norder && a.aligned) {
    const int row = a.order[q];
    if (tid == 0) issue(row, 0);
    if (tid < ntail) reinterpret_cast<uint16_t*>(buf_at(0))[tail0 + tid] = row_src(row)[tail0 + tid];
  }
  __syncthreads();
  int err = 0;

  for (int i = 0; q < a.norder; ++i) {
    const int row = a.order[q];
    unsigned long long* tr =
        a.trace ? a.trace + ((size_t)row * C + rank) * kTraceSlots : nullptr;
#define VT_RTRACE(k)                                      \
  do {                                                    \
    if (tr && tid == 0) tr[(k)] = global_timer_ns();      \
  } while (0)
    VT_RTRACE(0);
    const int b = i & 1, par = i & 1;
    const int qn = next_q(q + ncl);
    const int rown = qn < a.norder ? a.order[qn] : -1;
    uint16_t tail_v = 0;
    // the next row's slice into the other buffer, whose row ended with a barrier
    if (a.aligned && rown >= 0) {
      if (tid == 0) issue(rown, b ^ 1);
      if (tid < ntail) tail_v = row_src(rown)[tail0 + tid];  // stored at this row's end
    }
    if (a.aligned) {
      if (bulk && !mbar_wait_bounded(&s.full[b], (uint32_t)((i >> 1) & 1))) err |= kErrTimeout;
    } else {
      uint16_t* e = reinterpret_cast<uint16_t*>(buf_at(b));
      const uint16_t* src = row_src(row);
      for (int k = tid; k < nel; k += kRT) e[k] = src[k];
      __syncthreads();
    }
    const uint4* sv = reinterpret_cast<const uint4*>(buf_at(b));
    VT_RTRACE(1);

    const RowParams P = a.params[row];
    const bool greedy = (P.flags & kRowGreedy) != 0;
    const float inv_t = P.inv_t;
    float top_p = P.top_p;
    bool topp = (P.flags & kRowTopP) != 0;
    if (P.flags & kRowDecay) {  // the decayed top_p; 1 (the start) filters nothing
      top_p = a.decay[row].p;
      topp = top_p < 1.0f;
    }
    topp = topp && !greedy;
    const bool topk = !greedy && P.top_k > 1 && P.top_k < a.V;
    const bool minp = !greedy && (P.flags & kRowMinP) != 0;
    const bool filtered = topk || topp || minp;
    const bool need_hist = n > 0 || (!greedy && filtered);

    do {  // the row; `break` ends it
      // ---- pass A ----
      const Stats st = pass_stats(sv, vmax, nvec, lo, inv_t);
      {
        float m = st.rm, mt = st.rmt, sm = st.rs;
        int j = st.j, bad = st.bad ? 1 : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
          const int j2 = __shfl_xor_sync(0xffffffffu, j, o);
          const float mt2 = __shfl_xor_sync(0xffffffffu, mt, o);
          const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
          if (pair_better(m2, j2, m, j)) {
            m = m2;
            j = j2;
          }
          lse_combine(mt, sm, mt2, s2, kLog2e);
          bad |= __shfl_xor_sync(0xffffffffu, bad, o);
        }
        if (lane == 0) {
          s.rf[warp] = m;
          s.rf[kRW + warp] = mt;
          s.rf[2 * kRW + warp] = sm;
          s.ri[warp] = j;
          s.ri[kRW + warp] = bad;
        }
        __syncthreads();
        if (warp == 0) {
          float bm = lane < kRW ? s.rf[lane] : -INFINITY;
          float bmt = lane < kRW ? s.rf[kRW + lane] : -INFINITY;
          float bs = lane < kRW ? s.rf[2 * kRW + lane] : 0.f;
          int bj = lane < kRW ? s.ri[lane] : INT_MAX;
          int bb = lane < kRW ? s.ri[kRW + lane] : 0;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, bm, o);
            const int j2 = __shfl_xor_sync(0xffffffffu, bj, o);
            const float mt2 = __shfl_xor_sync(0xffffffffu, bmt, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, bs, o);
            if (pair_better(m2, j2, bm, bj)) {
              bm = m2;
              bj = j2;
            }
            lse_combine(bmt, bs, mt2, s2, kLog2e);
            bb |= __shfl_xor_sync(0xffffffffu, bb, o);
          }
          if (lane == 0) {
          RPart& pt = s.part[par];
          pt.xmax = bm;
          pt.s = bs;
          pt.arg = bj;
          pt.bad = bb || bm == INFINITY;
          pt.cmax = bm > -INFINITY ? bcode(__float_as_uint(bm) >> 16) : -bcode(0x7F80u);
          s.bf[0] = bmt;
          }
        }
        __syncthreads();
      }
      const int cmax_cta = s.part[par].cmax;
      const float mt_cta = s.bf[0];
      VT_RTRACE(2);

      // ---- thresholds and pass H ----
      int thr = kThrNone;
      unsigned int catch_cnt = 0;
      if (need_hist) {
        const int Kk = (topk && P.top_k <= kGrp * kRT) ? P.top_k : 0;
        int tn, tk;
        local_thresholds(st.gm, cmax_cta, n, Kk, s, &tn, &tk);
        if (greedy || !filtered) {
          thr = tn;
        } else {
          int tkept = topk ? (Kk > 0 ? tk : kThrAll) : kThrAll;
          if (minp) {
            if (warp == 0) {
              const int mc = mt_cta > -INFINITY ? minp_code_warp(inv_t, mt_cta, P.log_min_p, cmax_cta)
                                                : kThrAll;
              if (lane == 0) s.bi[6] = mc;
            }
            __syncthreads();
            tkept = max(tkept, s.bi[6]);
            __syncthreads();
          }
          thr = n > 0 ? min(tn, tkept) : tkept;
        }
        uint4* h4 = reinterpret_cast<uint4*>(hist);
        for (int k = tid; k < kSl / 4; k += kRT) h4[k] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        catch_cnt = (unsigned int)rblock_sum(
            (int)pass_counts(sv, vmax, nvec, code_floor_value(thr), cmax_cta, hist), s);
      }
      if (tid == 0) {
        RPart& pt = s.part[par];
        pt.thr = thr;
        pt.catch_cnt = catch_cnt;
        pt.err = err;
      }
      VT_RTRACE(3);
      cluster.sync();  // (1) statistics and histograms visible
      VT_RTRACE(4);

      // ---- the row's statistics from every CTA ----
      if (warp == 0) {
        float xm = -INFINITY, mt = -INFINITY, sm = 0.f;
        int arg = INT_MAX, bd = 0, th = INT_MIN, er = 0, cm = INT_MIN;
        unsigned int ct = 0u;
        if (lane < C) {
          const RPart* pp = cluster.map_shared_rank(&s.part[par], lane);
          xm = pp->xmax;
          mt = xm > -INFINITY ? __fmul_rn(xm, inv_t) : -INFINITY;
          sm = pp->s;
          arg = pp->arg;
          bd = pp->bad;
          th = pp->thr;
          ct = pp->catch_cnt;
          er = pp->err;
          cm = pp->cmax;
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
          bd |= __shfl_xor_sync(0xffffffffu, bd, o);
          er |= __shfl_xor_sync(0xffffffffu, er, o);
          th = max(th, __shfl_xor_sync(0xffffffffu, th, o));
          ct += __shfl_xor_sync(0xffffffffu, ct, o);
          cm = max(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        }
        if (lane < C) s.delta[lane] = cm - my_cmax;
        if (lane == 0) {
          s.bf[1] = xm;
          s.bf[2] = mt;
          s.bf[3] = sm;
          s.bi[0] = arg;
          s.bi[1] = bd || xm == INFINITY;
          s.bi[2] = th;
          s.bi[3] = (int)ct;
          s.bi[7] = er;
          s.bi[8] = cm;
        }
      }
      __syncthreads();
      const float xmax_row = s.bf[1], m_t = s.bf[2], S_row = s.bf[3];
      const int arg_row = s.bi[0], bad_row = s.bi[1], thr_row = s.bi[2];
      const unsigned int catch_tot = (unsigned int)s.bi[3];
      const int err_row = s.bi[7] | err, cmax_row = s.bi[8];
      const float lnS = logf(S_row);
      __syncthreads();
      const int status = bad_row ? kRowNonfinite : (xmax_row == -INFINITY ? kRowEmpty : kRowOk);

      if (status != kRowOk) {  // no token: -1, NaN log-probs; the seed still advances
        if (leader) {
          if (tid < n) {
            a.out_topk_ids[(int64_t)row * n + tid] = -1;
            a.out_topk_logprobs[(int64_t)row * n + tid] = __int_as_float(0x7fc00000);
          }
          if (tid == 0) {
            a.out_tokens[row] = -1;
            if (a.out_logprobs) a.out_logprobs[row] = __int_as_float(0x7fc00000);
            a.row_status[row] = status;
            a.dbg_kth_value[row] = __int_as_float(0x7fc00000);
            a.dbg_kth_index[row] = -1;
            a.dbg_kept[row] = 0;
            a.seeds[row] += kSeedStep;
            if (err_row) atomicOr(a.err_word, err_row);
          }
        }
        break;
      }
      if (greedy && n == 0) {  // the argmax, nothing else
        if (leader && tid == 0) {
          a.out_tokens[row] = arg_row;
          if (a.out_logprobs) a.out_logprobs[row] = -lnS;
          a.row_status[row] = kRowOk;
          a.dbg_kth_value[row] = m_t;
          a.dbg_kth_index[row] = arg_row;
          a.dbg_kept[row] = 1;
          a.seeds[row] += kSeedStep;
          if (err_row) atomicOr(a.err_word, err_row);
        }
        break;
      }

      // ---- the leader's walk (barrier 2), or every element kept ----
      const bool walk = need_hist;
      if (walk) {
        if (leader) {
          if (tid == 0) s.gcount = 0;
          WalkIn w;
          w.C = C;
          w.n = n;
          w.greedy = greedy;
          w.topk = topk;
          w.topp = topp;
          w.minp = minp;
          w.top_k = P.top_k;
          w.top_p = top_p;
          w.lmp = P.log_min_p;
          w.inv_t = inv_t;
          w.m_t = m_t;
          w.cmax = cmax_row;
          const long long Sstar = thr_row == kThrAll ? (long long)INT_MAX
                                                     : (long long)cmax_row - (long long)thr_row;
          w.full = Sstar >= kSlCatch;
          w.Smax = (int)(Sstar < kSlCatch - 1 ? Sstar : kSlCatch - 1);
          w.catch_tot = catch_tot;
          for (int r = 0; r < C; ++r) w.delta[r] = s.delta[r];
          leader_walk(w, hist, s);
          if (tid == 0 && s.res.action) {  // to the selection kernel, with the statistics
            SlowRow sr;
            sr.m_t = m_t;
            sr.lnS = lnS;
            sr.xmax = xmax_row;
            sr.bi_topn = (uint32_t)arg_row | (n == 0 ? 0x80000000u : 0u);
            a.slow[row] = sr;
            a.slow_list[atomicAdd(a.slow_ctl, 1u)] = row;
            if (err_row) atomicOr(a.err_word, err_row);
          }
        }
        VT_RTRACE(5);
        cluster.sync();  // (2) the walk visible
        VT_RTRACE(6);
        if (tid < (int)(sizeof(RRes) / 4)) {
          const int* src = reinterpret_cast<const int*>(cluster.map_shared_rank(&s.res, 0));
          reinterpret_cast<int*>(&s.rl)[tid] = src[tid];
        }
        __syncthreads();
        if (s.rl.action) break;
      } else {
        if (tid == 0) {
          s.rl.action = 0;
          s.rl.beta = kAllKept;
          s.rl.sn = -1;
          s.rl.L3 = 0;
          s.rl.last_rank = -1;
          s.rl.cb[rank] = s.rl.nb[rank] = s.rl.cn[rank] = s.rl.nn[rank] = 0;
        }
        __syncthreads();
      }

      // ---- pass D: the draw over the kept elements, the top-n to the leader ----
      // Slot S < beta holds values above x_b = value(beta) (codes are
      // monotone; beta is never the code-0 slot), so the tests are value
      // compares: kept iff x > x_b, or x == x_b and among the first cb of the
      // boundary slot here; likewise the top-n against x_n.  Vectors whose
      // maximum is below both are skipped whole.
      const int beta = s.rl.beta, sn = s.rl.sn;
      const int cb = s.rl.cb[rank], nb = s.rl.nb[rank];
      const int cnq = s.rl.cn[rank], nnq = s.rl.nn[rank];
      const bool bfull = cb == nb, nfull = cnq == nnq;
      const bool keep_all = beta == kAllKept;
      const float xb = beta >= 0 ? bcode_value(cmax_row - beta) : INFINITY;
      const float xn = sn >= 0 ? bcode_value(cmax_row - sn) : INFINITY;
      const float lim = keep_all ? -INFINITY : fminf(xb, xn);
      const uint64_t key = row_key(a.seeds[row], row);
      if (tid == 0) {
        s.nlist = 0;
        s.nlistn = 0;
      }
      __syncthreads();
      int* gc = cluster.map_shared_rank(&s.gcount, 0);
      uint64_t* gb = cluster.map_shared_rank(s.gather, 0);
      auto push = [&](float x, int j) {
        const int pos = atomicAdd(gc, 1);
        if (pos < kGatherCap) gb[pos] = elem_key(__fmul_rn(x, inv_t), (uint32_t)j);
      };
      float bs = -INFINITY, bz = 0.f;
      int bj = INT_MAX, kthmax = -1, fin = 0;
      unsigned long long lastk = ~0ull;
      // Noise prefilter: an element beats the running best bs only if
      // -ln u < e^(z - bs) <= e^(m_t - bs) = E, and -ln u >= 1 - u, so only if
      // u > 1 - E: 24-bit noise b >= blo (a 2^-8 margin and one unit cover
      // the fp32 rounding).  Those pass to the per-element certificate.
      uint32_t blo = 0u;
      auto set_blo = [&]() {
        const float E = ex2_approx(__fmul_rn(__fsub_rn(m_t, bs), kLog2e)) * 1.00390625f;
        const float th = (1.0f - E) * 16777216.0f;
        blo = (E < 1.0f && th > 1.0f) ? (uint32_t)th - 1u : 0u;
      };
      auto consider = [&](float x, int j, uint32_t bits) {
        if (bits < blo) return;
        const float z = __fmul_rn(x, inv_t);
        if (!may_beat(z, bs, bits)) return;
        const float sc = gumbel_score(z, bits);
        if (pair_better(sc, j, bs, bj)) {
          bs = sc;
          bj = j;
          bz = z;
          set_blo();
        }
      };
      for (int v = tid; v < nvec; v += kRT) {
        if (!(__uint_as_float((uint32_t)vmax[v] << 16) >= lim)) continue;
        const uint4 qv = sv[v];
        float x[8];
        unpack8(qv, x);
        uint32_t km = 0u, rare = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const bool fin_i = x[i] > -INFINITY;
          const bool kp = keep_all ? fin_i : x[i] > xb;
          km |= (uint32_t)kp << i;
          rare |= (uint32_t)(x[i] == xb || x[i] >= xn) << i;
        }
        if (keep_all) {
          fin += __popc(km);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (km & (1u << i)) {
              const unsigned long long k =
                  elem_key(__fmul_rn(x[i], inv_t), (uint32_t)(lo + 8 * v + i));
              lastk = k < lastk ? k : lastk;
            }
          }
        }
        while (rare) {  // top-n members and boundary-slot elements (few)
          const int i = __ffs(rare) - 1;
          rare &= rare - 1u;
          const int j = lo + 8 * v + i;
          const float xe = __uint_as_float(bits8(qv, i) << 16);
          if (xe > xn || (xe == xn && nfull)) {
            push(xe, j);
          } else if (xe == xn && cnq > 0) {
            const int pos = atomicAdd(&s.nlistn, 1);
            if (pos < kListCap) list_n[pos] = (uint32_t)(j - lo);
          }
          if (xe == xb) {
            if (bfull) {
              km |= 1u << i;
              kthmax = max(kthmax, j);
            } else if (cb > 0) {
              const int pos = atomicAdd(&s.nlist, 1);
              if (pos < kListCap) list_b[pos] = (uint32_t)(j - lo);
            }
          }
        }
        if (km) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            if (km & (3u << (2 * w))) {
              const int j0 = lo + 8 * v + 2 * w;
              const uint64_t h = pair_hash(key, j0);
              if (km & (1u << (2 * w))) consider(x[2 * w], j0, bits_even(h));
              if (km & (2u << (2 * w))) consider(x[2 * w + 1], j0 + 1, bits_odd(h));
            }
          }
        }
      }
      __syncthreads();
      // the kept (top-n) part of a boundary slot: its lowest indices here
      const int nl = s.nlist, nln = s.nlistn;
      const uint16_t* e16 = reinterpret_cast<const uint16_t*>(buf_at(b));
      if (beta >= 0 && cb > 0 && cb < nb) {
        if (nl != nb && tid == 0) err |= kErrInternal;
        const uint32_t kth = rblock_kth_smallest(list_b, min(nl, kListCap), cb, hist, s);
        for (int e = tid; e < min(nl, kListCap); e += kRT) {
          const uint32_t off = list_b[e];
          if (off <= kth) {
            const int j = lo + (int)off;
            consider(__uint_as_float((uint32_t)e16[off] << 16), j, noise_bits(key, j));
          }
        }
        if (tid == 0) kthmax = max(kthmax, lo + (int)kth);
      }
      if (sn >= 0 && cnq > 0 && cnq < nnq) {
        if (nln != nnq && tid == 0) err |= kErrInternal;
        const uint32_t kth = rblock_kth_smallest(list_n, min(nln, kListCap), cnq, hist, s);
        for (int e = tid; e < min(nln, kListCap); e += kRT) {
          const uint32_t off = list_n[e];
          if (off <= kth) push(__uint_as_float((uint32_t)e16[off] << 16), lo + (int)off);
        }
      }
      VT_RTRACE(7);
      rblock_argmax(bs, bj, bz, s);
      kthmax = rblock_max(kthmax, s);
      if (beta == kAllKept) {
        lastk = rblock_min_u64(lastk, s);
        fin = rblock_sum(fin, s);
      }
      if (tid == 0) {
        RPart& pt = s.part[par];
        pt.best_s = bs;
        pt.best_j = bj;
        pt.best_z = bz;
        pt.kth_j = rank == s.rl.last_rank ? kthmax : -1;
        pt.last_key = lastk;
        pt.fin = fin;
        pt.err = err;
      }
      VT_RTRACE(8);
      cluster.sync();  // (3) draw partials and the top-n keys visible
      VT_RTRACE(9);

      // ---- the leader writes the row ----
      if (leader) {
        if (warp == 0) {  // lanes < C read the CTAs' draw partials
          float best = -INFINITY, bzz = 0.f;
          int bjj = INT_MAX, nfin = 0, er = 0, kjr = -1;
          unsigned long long lk = ~0ull;
          if (lane < C) {
            const RPart* pp = cluster.map_shared_rank(&s.part[par], lane);
            best = pp->best_s;
            bjj = pp->best_j;
            bzz = pp->best_z;
            lk = pp->last_key;
            nfin = pp->fin;
            er = pp->err;
            kjr = lane == s.rl.last_rank ? pp->kth_j : -1;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
            const int j2 = __shfl_xor_sync(0xffffffffu, bjj, o);
            const float z2 = __shfl_xor_sync(0xffffffffu, bzz, o);
            if (pair_better(b2, j2, best, bjj)) {
              best = b2;
              bjj = j2;
              bzz = z2;
            }
            const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, lk, o);
            lk = l2 < lk ? l2 : lk;
            nfin += __shfl_xor_sync(0xffffffffu, nfin, o);
            er |= __shfl_xor_sync(0xffffffffu, er, o);
            kjr = max(kjr, __shfl_xor_sync(0xffffffffu, kjr, o));
          }
          if (lane == 0) {
            int tok = arg_row, kj = arg_row, L3 = 1;
            float ztok = m_t, kz = m_t;
            er |= err_row;
            if (!greedy) {
              tok = bjj;
              ztok = bzz;
              if (beta >= 0) {
                kz = s.rl.kth_z;
                kj = kjr;
                L3 = s.rl.L3;
              } else {
                kz = key_z(lk);
                kj = (int)key_idx(lk);
                L3 = nfin;
              }
              if (tok == INT_MAX || kj < 0) er |= kErrInternal;
            }
            if (n > 0 && s.gcount != n) er |= kErrInternal;
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
            if (er) atomicOr(a.err_word, er);
          }
        }
        if (n > 0 && warp == 0) {  // the top-n, ordered (value desc, index asc)
          const int g = min(s.gcount, kGatherCap);
          const uint64_t k = lane < g ? s.gather[lane] : 0ull;
          int rk = 0;
          for (int t = 0; t < g; ++t) rk += s.gather[t] > k;
          if (lane < g && rk < n) {
            a.out_topk_ids[(int64_t)row * n + rk] = (int)key_idx(k);
            a.out_topk_logprobs[(int64_t)row * n + rk] = (key_z(k) - m_t) - lnS;
          }
        }
      }
    } while (0);
    VT_RTRACE(10);
#undef VT_RTRACE

    // ---- row end: the next row's last elements, then its buffer is complete ----
    if (a.aligned && rown >= 0 && tid < ntail)
      reinterpret_cast<uint16_t*>(buf_at(b ^ 1))[tail0 + tid] = tail_v;
    __syncthreads();
    q = qn;
  }
  if (err) atomicOr(a.err_word, err);
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace
}  // namespace vt

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace vt {

RowPlan plan_rows(int B, int V) {
  RowPlan p{};
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return p;
  const size_t fixed = (size_t)kSl * 4 + (size_t)2 * kListCap * 4;
  const size_t room = (size_t)optin > sizeof(RSmem) ? (size_t)optin - sizeof(RSmem) : 0;
  for (int C = 1; C <= kRMaxC; C <<= 1) {
    int slice = (V + C - 1) / C;
    slice = (slice + 7) & ~7;
    const uint32_t buf = (uint32_t)(((size_t)slice * 2 + 127) & ~(size_t)127);
    const size_t smem = 2 * (size_t)buf + fixed + (((size_t)slice / 8 * 2 + 15) & ~(size_t)15);
    if (smem > room) continue;
    cudaError_t e = cudaFuncSetAttribute(rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(rows_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return p;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, 1, 1);
    cfg.blockDim = dim3(kRT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, rows_kernel, &cfg) != cudaSuccess ||
        nclusters < 1) {
      (void)cudaGetLastError();
      continue;
    }
    p.cluster = C;
    p.slice = slice;
    p.buf_bytes = buf;
    p.smem = smem;
    p.clusters = nclusters < B ? nclusters : B;
    return p;
  }
  return p;
}

cudaError_t launch_rows(const RowArgs& args, const RowPlan& plan, cudaStream_t stream) {
  if (plan.cluster < 1 || plan.clusters < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(plan.clusters * plan.cluster), 1, 1);
  cfg.blockDim = dim3(kRT, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rows_kernel, args);
}

}  // namespace vt
