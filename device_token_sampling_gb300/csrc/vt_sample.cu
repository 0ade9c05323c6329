// vt_sample.cu -- the fused batched decode sampling kernel for sm_103a.
//
// One thread-block cluster per logits row.  Each CTA of the cluster owns one
// contiguous slice of the row, stages it ONCE in shared memory with bulk
// asynchronous copies (cp.async.bulk, completion on an mbarrier), and runs
// every pass of the pipeline over shared memory; HBM sees each logit once.
// Cross-CTA results move through distributed shared memory (DSMEM) between
// hardware cluster barriers, so no CTA ever spins on another.
//
// Pipeline per row (pages: TensorRT-LLM "Sampling" for the penalty, temperature
// and filter formulas; vllm.cpp's Gumbel-draw pull request for the seeded
// draw and the lowest-index ArgReduce; the Tenstorrent sampling README for the
// log-softmax and the reset-then-sample state):
//   1. penalties: the row's (id, count) table entries that fall in the slice
//      are rewritten (repetition, frequency, presence) into a side list and
//      masked out of the dense slice;
//   2. pass A: row max, online sum of exp, lowest-index argmax, per-group and
//      per-thread maxima (temperature folded into one FFMA per element);
//   3. candidates: a threshold that provably admits at least K elements
//      (the K/C-th largest per-thread maximum of each CTA, minimum over the
//      cluster) collects a prefix of the order (value desc, index asc) into
//      the leader CTA, which sorts it and applies min-p, top-k and top-p
//      without touching the rest of the row;
//   4. when the kept set is not inside the candidates (a wide top-p nucleus,
//      a large top-k, an unfiltered draw), a cluster-wide radix select on
//      64-bit (value, index) keys with count/mass histograms finds the exact
//      boundary, and a draw pass scores only elements that can still win
//      (a 1 - u >= exp(z - s) certificate skips the logarithms);
//   5. outputs: token, its log-prob, top-n log-probs, row status, the kept
//      boundary, the seed advance and the optional count append.
#include "vt_device.cuh"
#include "vt_kernels.h"

#include <climits>

namespace cg = cooperative_groups;

namespace vt {
namespace {

constexpr int kGatherCap = 2048;    // keys the leader CTA can hold and sort
constexpr int kBinBits = 10;
constexpr int kBins = 1 << kBinBits;
constexpr int kDefaultCand = 512;   // candidates tried for top-p / min-p rows
constexpr int kGroupBytes = 32;     // one thread step: two 16-byte vectors
constexpr uint32_t kBulkChunk = 32768;
constexpr int kMaxCluster = 16;

// Row status codes (match VT_ROW_* in the public header).
constexpr int kRowOk = 0, kRowNonfinite = 1, kRowEmpty = 2, kRowHistoryFull = 3;

template <typename T>
struct Elt;

template <>
struct Elt<float> {
  static constexpr int kPerGroup = kGroupBytes / 4;
  __device__ static void load(const float* d, int g, float* x) {
    const uint4* p = reinterpret_cast<const uint4*>(d + g * kPerGroup);
    const uint4 a = p[0], b = p[1];
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  }
  __device__ static float at(const float* d, int e) { return d[e]; }
  __device__ static void mask(float* d, int e) { d[e] = -INFINITY; }
  __device__ static void copy_global(float* d, int e, const float* row, int64_t j) {
    d[e] = __ldg(row + j);
  }
  __device__ static void fill_neg_inf(float* d, int e) { d[e] = -INFINITY; }
};

// bfloat16 stored as its 16 bits; widening to fp32 is exact (a 16-bit shift).
template <>
struct Elt<uint16_t> {
  static constexpr int kPerGroup = kGroupBytes / 2;
  __device__ static void load(const uint16_t* d, int g, float* x) {
    const uint4* p = reinterpret_cast<const uint4*>(d + g * kPerGroup);
    const uint4 a = p[0], b = p[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static float at(const uint16_t* d, int e) {
    return __uint_as_float((uint32_t)d[e] << 16);
  }
  __device__ static void mask(uint16_t* d, int e) { d[e] = 0xFF80u; }
  __device__ static void copy_global(uint16_t* d, int e, const uint16_t* row, int64_t j) {
    d[e] = __ldg(row + j);
  }
  __device__ static void fill_neg_inf(uint16_t* d, int e) { d[e] = 0xFF80u; }
};

// Per-CTA partial results; other CTAs of the cluster read them over DSMEM.
struct Part {
  float m, s, bv;
  int bi;
  int nonfinite;
  float tau;
  int ncand, ncand_minp;
  unsigned long long cand_mass;
  unsigned long long rng_cnt, rng_mass;
  float dscore, dz;
  int didx;
  int kept;
  unsigned long long kmin;
  float s_exact;
  int err;
};

// Row-level values every CTA derives identically from the partials.
struct RowStats {
  float M, S, m_t, lnS, bv;
  int bi;
  int nonfinite;
  float tau;
  int nc, nc_minp;
  unsigned long long cand_mass;
  int err;
};

// Selection result, written by the leader and read by every CTA.
struct SelOut {
  unsigned long long kb, cnt_incl, mass_incl, total_cnt, total_mass;
  int all;
};

// Digit walk of one selection level (identical in every CTA).
struct Walk {
  int d;
  int found;
  unsigned long long acc_c, acc_m, band_cnt, total_c, total_m;
};

struct __align__(16) Smem {
  uint64_t mbar;
  Part part;
  RowStats rs;
  SelOut sel;
  Walk walk;
  int gcount;
  int e_lo, e_hi;
  int bcast_i[4];
  float bcast_f[4];
  unsigned long long bcast_u[4];
  float tmax[kThreads];
  float rf[kWarps * 4];
  int ri[kWarps * 4];
  unsigned long long ru[kWarps * 4];
};

struct Ctx {
  int tid, lane, warp;
  int C, rank, row, V, lo, hi, slice, ngroups;
  float inv_t, ax;     // 1/T and log2(e)/T
  float m_t, lnS;      // row max of z_t, ln(sum exp(z_t - m_t))
  bool greedy, topk, topp, minp;
  int top_k;
  float top_p;
  double lmp;          // ln(min_p)
  float* gmax;         // per group max of the pre-temperature values
  uint64_t* gather;    // leader key buffer (this CTA's copy)
  unsigned int* hcnt;  // selection histograms (alias the gather buffer)
  unsigned long long* hmass;
  unsigned int* mcnt;  // merged bins of this CTA's digit range
  unsigned long long* mmass;
  const int2* tab;     // this row's count table
  const float* zs;     // penalised values of the table entries
  int e_lo, e_hi;      // table entries inside the slice
  uint64_t rkey;       // noise stream key
};

// ---------------------------------------------------------------------------
// block-level helpers (all threads of the CTA must call them)
// ---------------------------------------------------------------------------
__device__ int block_sum_int(int v, Smem& s) {
  v = warp_sum_i(v);
  if ((threadIdx.x & 31) == 0) s.ri[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int t = threadIdx.x < kWarps ? s.ri[threadIdx.x] : 0;
    t = warp_sum_i(t);
    if (threadIdx.x == 0) s.ri[kWarps] = t;
  }
  __syncthreads();
  const int r = s.ri[kWarps];
  __syncthreads();
  return r;
}

__device__ float block_sum_f(float v, Smem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) s.rf[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += s.rf[w];
    s.rf[kWarps] = t;
  }
  __syncthreads();
  const float r = s.rf[kWarps];
  __syncthreads();
  return r;
}

__device__ unsigned long long block_sum_u64(unsigned long long v, Smem& s) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < kWarps ? s.ru[threadIdx.x] : 0ull;
    t = warp_sum_u64(t);
    if (threadIdx.x == 0) s.ru[kWarps] = t;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kWarps];
  __syncthreads();
  return r;
}

__device__ unsigned long long block_min_u64(unsigned long long v, Smem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w < v ? w : v;
  }
  if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < kWarps ? s.ru[threadIdx.x] : ~0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long w = __shfl_xor_sync(0xffffffffu, t, o);
      t = w < t ? w : t;
    }
    if (threadIdx.x == 0) s.ru[kWarps] = t;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kWarps];
  __syncthreads();
  return r;
}

// Exclusive prefix of one u64 per thread over the CTA; *total gets the sum.
__device__ unsigned long long block_exclusive_u64(unsigned long long v, Smem& s,
                                                  unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long w = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += w;
  }
  if (lane == 31) s.ru[warp] = inc;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < kWarps ? s.ru[threadIdx.x] : 0ull;
    unsigned long long ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long w = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += w;
    }
    if (threadIdx.x < kWarps) s.ru[kWarps + threadIdx.x] = ti - t;
    if (threadIdx.x == kWarps - 1) s.ru[2 * kWarps] = ti;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kWarps + warp] + inc - v;
  *total = s.ru[2 * kWarps];
  __syncthreads();
  return r;
}

// (score, index, payload) argmax over the CTA; larger score, then lower index.
__device__ void block_argmax(float& v, int& i, float& z, Smem& s) {
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
    s.rf[kWarps + warp] = z;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float tv = lane < kWarps ? s.rf[lane] : -INFINITY;
    int ti = lane < kWarps ? s.ri[lane] : INT_MAX;
    float tz = lane < kWarps ? s.rf[kWarps + lane] : 0.f;
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
    if (threadIdx.x == 0) {
      s.rf[2 * kWarps] = tv;
      s.ri[2 * kWarps] = ti;
      s.rf[2 * kWarps + 1] = tz;
    }
  }
  __syncthreads();
  v = s.rf[2 * kWarps];
  i = s.ri[2 * kWarps];
  z = s.rf[2 * kWarps + 1];
  __syncthreads();
}

// Bitonic sort, descending, of n (a power of two) keys in shared memory.
__device__ void bitonic_desc_u64(uint64_t* keys, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__device__ void bitonic_desc_f32(float* v, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const float a = v[i], b = v[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            v[i] = b;
            v[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ int pow2_ceil(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// min-p test z_t - m >= ln(min_p), decided exactly in double; fp32 decides
// whenever it is far from the threshold.
__device__ __forceinline__ bool minp_pass(float zt, float m_t, double lmp) {
  const float d = zt - m_t;
  const float l = (float)lmp;
  const float margin = 1e-4f * (1.0f + fabsf(l));
  if (d > l + margin) return true;
  if (d < l - margin) return false;
  return (double)zt - (double)m_t >= lmp;
}

// Occurrence penalties of one seen token: repetition, frequency, presence
// (fp32, each operation rounded once).
__device__ __forceinline__ float penalize(float x, int count, const RowParams& P) {
  float z = x;
  if (P.repetition != 1.0f)
    z = (z >= 0.0f) ? __fdiv_rn(z, P.repetition) : __fmul_rn(z, P.repetition);
  z = __fsub_rn(z, __fmul_rn(P.frequency, (float)count));
  z = __fsub_rn(z, P.presence);
  return z;
}

// Does this dense slot hold a penalised token (whose value lives in the side
// list instead)?  Binary search of the slice's table entries.
__device__ bool is_side_slot(const Ctx& c, int j) {
  int a = c.e_lo, b = c.e_hi;
  while (a < b) {
    const int mid = (a + b) >> 1;
    const int id = c.tab[mid].x;
    if (id == j) return true;
    if (id < j) a = mid + 1; else b = mid;
  }
  return false;
}

// Visit every element of the slice: dense groups whose max passes
// `group_ok(fl(gmax * inv_t))`, then the side list.  elem(zt, j) gets the
// tempered value and the global index.
template <typename T, typename GF, typename EF>
__device__ __forceinline__ void for_each_elem(const Ctx& c, const T* data, GF group_ok,
                                              EF elem) {
  constexpr int E = Elt<T>::kPerGroup;
  for (int g = c.tid; g < c.ngroups; g += kThreads) {
    if (!group_ok(c.gmax[g] * c.inv_t)) continue;
    float x[E];
    Elt<T>::load(data, g, x);
    const int j0 = c.lo + g * E;
#pragma unroll
    for (int i = 0; i < E; ++i) elem(x[i] * c.inv_t, j0 + i, false);
  }
  for (int e = c.e_lo + c.tid; e < c.e_hi; e += kThreads)
    elem(c.zs[e] * c.inv_t, c.tab[e].x, true);
}

// ---------------------------------------------------------------------------
// cluster-wide radix selection on (value, index) keys
// ---------------------------------------------------------------------------
enum Pred { kPredAll = 0, kPredSurv = 1 };

// Find the first element, in the order (value desc, index asc), of the set
// {pred, key >= kbound} whose inclusive count exceeds `count_target`
// (by_mass = false) or whose inclusive mass exceeds p * (mass of the set)
// (by_mass = true).  Every CTA of the cluster calls it with identical
// arguments and receives the same result.
template <typename T>
__device__ SelOut cluster_select(Ctx& c, const T* data, Smem& s, cg::cluster_group& cluster,
                                 int pred, unsigned long long kbound, bool by_mass,
                                 unsigned long long count_target, float p) {
  unsigned long long Klo = kbound, Khi = ~0ull;
  unsigned long long acc_c = 0, acc_m = 0;
  unsigned long long target = count_target;
  unsigned long long total_c = 0, total_m = 0;
  bool first = true;
  SelOut out;
  out.all = 0;
  const int b0 = c.rank * (kBins / c.C), nb = kBins / c.C;

  auto in_pred = [&](float zt, int j, bool side) -> bool {
    if (pred == kPredAll) {
      if (j >= c.V) return false;
      if (zt == -INFINITY && !side && is_side_slot(c, j)) return false;
      return true;
    }
    if (!(zt > -INFINITY)) return false;
    return !c.minp || minp_pass(zt, c.m_t, c.lmp);
  };

  for (int level = 0; level < 8; ++level) {
    const unsigned long long range = Khi - Klo;
    const int bits = range == 0 ? 0 : 64 - __clzll((long long)range);
    const int shift = bits > kBinBits ? bits - kBinBits : 0;
    for (int b = c.tid; b < kBins; b += kThreads) {
      c.hcnt[b] = 0u;
      c.hmass[b] = 0ull;
    }
    __syncthreads();
    const uint32_t klo_hi = (uint32_t)(Klo >> 32);
    for_each_elem<T>(
        c, data, [&](float gz) { return ord_key(gz) >= klo_hi; },
        [&](float zt, int j, bool side) {
          if (!in_pred(zt, j, side)) return;
          const unsigned long long K = elem_key(zt, (uint32_t)j);
          if (K < Klo || K > Khi) return;
          const int d = (int)((Khi - K) >> shift);
          atomicAdd(&c.hcnt[d], 1u);
          if (by_mass) atomicAdd(&c.hmass[d], mass_fixed(zt, c.m_t));
        });
    cluster.sync();
    // distributed merge: this CTA sums its digit range over the cluster
    unsigned long long my_c = 0, my_m = 0;
    for (int b = c.tid; b < nb; b += kThreads) {
      unsigned long long sc = 0, sm = 0;
      for (int r = 0; r < c.C; ++r) {
        const unsigned int* rc = cluster.map_shared_rank(c.hcnt, r);
        const unsigned long long* rm = cluster.map_shared_rank(c.hmass, r);
        sc += rc[b0 + b];
        sm += rm[b0 + b];
      }
      c.mcnt[b] = (unsigned int)sc;
      c.mmass[b] = sm;
      my_c += sc;
      my_m += sm;
    }
    my_c = block_sum_u64(my_c, s);
    my_m = block_sum_u64(my_m, s);
    if (c.tid == 0) {
      s.part.rng_cnt = my_c;
      s.part.rng_mass = my_m;
    }
    cluster.sync();
    // walk: warp 0 finds the range, then the digit (identical in every CTA)
    if (c.warp == 0) {
      unsigned long long rc = 0, rm = 0;
      if (c.lane < c.C) {
        const Part* pr = cluster.map_shared_rank(&s.part, c.lane);
        rc = pr->rng_cnt;
        rm = pr->rng_mass;
      }
      unsigned long long ic = rc, im = rm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long wc = __shfl_up_sync(0xffffffffu, ic, o);
        const unsigned long long wm = __shfl_up_sync(0xffffffffu, im, o);
        if (c.lane >= o) {
          ic += wc;
          im += wm;
        }
      }
      const unsigned long long tc = __shfl_sync(0xffffffffu, ic, 31);
      const unsigned long long tm = __shfl_sync(0xffffffffu, im, 31);
      if (c.lane == 0) {
        s.walk.total_c = tc;
        s.walk.total_m = tm;
      }
      unsigned long long tgt = target;
      if (first && by_mass) tgt = (unsigned long long)((double)tm * (double)p);
      // first range whose inclusive cumulative value exceeds the target
      const unsigned long long base_c = acc_c, base_m = acc_m;
      const bool cross = c.lane < c.C &&
                         (by_mass ? (base_m + im > tgt) : (base_c + ic > tgt));
      const unsigned int mask = __ballot_sync(0xffffffffu, cross);
      if (c.lane == 0) {
        s.walk.found = mask != 0;
        s.bcast_u[0] = tgt;
      }
      if (mask != 0) {
        const int r = __ffs(mask) - 1;
        const unsigned long long before_c = base_c + __shfl_sync(0xffffffffu, ic - rc, r);
        const unsigned long long before_m = base_m + __shfl_sync(0xffffffffu, im - rm, r);
        // digits of range r live in CTA r's merged arrays
        const unsigned int* mc = cluster.map_shared_rank(c.mcnt, r);
        const unsigned long long* mm = cluster.map_shared_rank(c.mmass, r);
        unsigned long long run_c = before_c, run_m = before_m;
        int dsel = -1;
        unsigned long long sel_c = 0, sel_m = 0, band = 0;
        for (int base = 0; base < nb && dsel < 0; base += 32) {
          const int b = base + c.lane;
          const unsigned long long vc = b < nb ? mc[b] : 0ull;
          const unsigned long long vm = b < nb ? mm[b] : 0ull;
          unsigned long long xc = vc, xm = vm;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long wc = __shfl_up_sync(0xffffffffu, xc, o);
            const unsigned long long wm = __shfl_up_sync(0xffffffffu, xm, o);
            if (c.lane >= o) {
              xc += wc;
              xm += wm;
            }
          }
          const bool hit = b < nb && (by_mass ? (run_m + xm > tgt) : (run_c + xc > tgt));
          const unsigned int hm = __ballot_sync(0xffffffffu, hit);
          if (hm != 0) {
            const int l = __ffs(hm) - 1;
            dsel = r * nb + base + l;
            sel_c = run_c + __shfl_sync(0xffffffffu, xc - vc, l);
            sel_m = run_m + __shfl_sync(0xffffffffu, xm - vm, l);
            band = __shfl_sync(0xffffffffu, vc, l);
          } else {
            run_c += __shfl_sync(0xffffffffu, xc, 31);
            run_m += __shfl_sync(0xffffffffu, xm, 31);
          }
        }
        if (c.lane == 0) {
          s.walk.d = dsel;
          s.walk.acc_c = sel_c;
          s.walk.acc_m = sel_m;
          s.walk.band_cnt = band;
        }
      }
    }
    __syncthreads();
    if (first) {
      total_c = s.walk.total_c;
      total_m = s.walk.total_m;
      target = s.bcast_u[0];
      first = false;
    }
    const bool found = s.walk.found;
    const int d = s.walk.d;
    const unsigned long long band = s.walk.band_cnt;
    acc_c = s.walk.acc_c;
    acc_m = s.walk.acc_m;
    if (c.rank == 0 && c.tid == 0) s.gcount = 0;
    cluster.sync();  // merged arrays and parts are free again
    if (!found) {
      out.all = 1;
      out.kb = kbound;
      out.cnt_incl = total_c;
      out.mass_incl = total_m;
      out.total_cnt = total_c;
      out.total_mass = total_m;
      return out;
    }
    // narrow the key range to digit d
    const unsigned long long hi_new = Khi - ((unsigned long long)d << shift);
    const unsigned long long width = shift >= 64 ? ~0ull : ((1ull << shift) - 1ull);
    const unsigned long long lo_new = (hi_new - Klo > width) ? hi_new - width : Klo;
    Khi = hi_new;
    Klo = lo_new;
    if (band <= (unsigned long long)kGatherCap || Klo == Khi) break;
  }
  // collect the band into the leader, sort it, and walk it
  {
    uint64_t* lg = cluster.map_shared_rank(c.gather, 0);
    int* lcount = cluster.map_shared_rank(&s.gcount, 0);
    const uint32_t klo_hi = (uint32_t)(Klo >> 32);
    for_each_elem<T>(
        c, data, [&](float gz) { return ord_key(gz) >= klo_hi; },
        [&](float zt, int j, bool side) {
          if (!in_pred(zt, j, side)) return;
          const unsigned long long K = elem_key(zt, (uint32_t)j);
          if (K < Klo || K > Khi) return;
          const int pos = atomicAdd(lcount, 1);
          if (pos < kGatherCap) lg[pos] = K;
        });
    cluster.sync();
    if (c.rank == 0) {
      const int n = min(s.gcount, kGatherCap);
      const int P2 = pow2_ceil(max(n, 1));
      for (int i = n + c.tid; i < P2; i += kThreads) c.gather[i] = 0ull;
      __syncthreads();
      bitonic_desc_u64(c.gather, P2);
      // chunked inclusive scan of the band, first crossing position
      const int per = (n + kThreads - 1) / kThreads;
      const int i0 = c.tid * per, i1 = min(n, i0 + per);
      unsigned long long lc = 0, lm = 0;
      for (int i = i0; i < i1; ++i) {
        lc += 1;
        if (by_mass) lm += mass_fixed(key_z(c.gather[i]), c.m_t);
      }
      unsigned long long tot;
      const unsigned long long ex_c = block_exclusive_u64(lc, s, &tot);
      const unsigned long long ex_m = block_exclusive_u64(lm, s, &tot);
      int hit = INT_MAX;
      unsigned long long hit_c = 0, hit_m = 0;
      unsigned long long rc = acc_c + ex_c, rm = acc_m + ex_m;
      for (int i = i0; i < i1; ++i) {
        rc += 1;
        if (by_mass) rm += mass_fixed(key_z(c.gather[i]), c.m_t);
        if (by_mass ? (rm > target) : (rc > target)) {
          hit = i;
          hit_c = rc;
          hit_m = rm;
          break;
        }
      }
      // lowest crossing position over the CTA
      int hmin = hit;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) hmin = min(hmin, __shfl_xor_sync(0xffffffffu, hmin, o));
      if (c.lane == 0) s.ri[c.warp] = hmin;
      __syncthreads();
      if (c.tid == 0) {
        int h = INT_MAX;
        for (int w = 0; w < kWarps; ++w) h = min(h, s.ri[w]);
        s.bcast_i[0] = h;
      }
      __syncthreads();
      const int h = s.bcast_i[0];
      if (h != INT_MAX && hit == h) {
        s.sel.kb = c.gather[h];
        s.sel.cnt_incl = hit_c;
        s.sel.mass_incl = hit_m;
        s.sel.all = 0;
      }
      if (h == INT_MAX && c.tid == 0) {  // cannot happen: the band holds the crossing
        s.sel.kb = n > 0 ? c.gather[n - 1] : kbound;
        s.sel.cnt_incl = acc_c + n;
        s.sel.mass_incl = acc_m;
        s.sel.all = 0;
        atomicOr(&s.part.err, kErrInternal);
      }
      if (c.tid == 0) {
        s.sel.total_cnt = total_c;
        s.sel.total_mass = total_m;
      }
    }
    cluster.sync();
    const SelOut* ls = cluster.map_shared_rank(&s.sel, 0);
    out = *ls;
    __syncthreads();
    cluster.sync();  // the leader's buffers may be reused after this
  }
  return out;
}

// ---------------------------------------------------------------------------
// count-table append (leader CTA, after the draw)
// ---------------------------------------------------------------------------
__device__ void append_token(int2* tab, int32_t* len_p, int cap, int tok, Smem& s,
                             int32_t* status_p) {
  const int len = *len_p;
  int below = 0;
  for (int e = threadIdx.x; e < len; e += kThreads) below += tab[e].x < tok;
  const int pos = block_sum_int(below, s);
  const bool exists = pos < len && tab[pos].x == tok;
  if (exists) {
    if (threadIdx.x == 0) tab[pos].y += 1;
    return;
  }
  if (len >= cap) {
    if (threadIdx.x == 0) *status_p = kRowHistoryFull;
    return;
  }
  // shift [pos, len) up by one, highest chunk first
  for (int top = len; top > pos; top -= kThreads) {
    const int e = top - 1 - threadIdx.x;
    int2 v = make_int2(0, 0);
    const bool mine = e >= pos && e >= top - kThreads;
    if (mine) v = tab[e];
    __syncthreads();
    if (mine) tab[e + 1] = v;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    tab[pos] = make_int2(tok, 1);
    *len_p = len + 1;
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ Smem s;
  cg::cluster_group cluster = cg::this_cluster();

  Ctx c;
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  c.C = (int)cluster_nctarank();
  c.rank = (int)cluster_ctarank();
  c.row = blockIdx.x / c.C;
  c.V = a.V;
  c.slice = a.slice;
  c.lo = c.rank * a.slice;
  c.hi = min(c.lo + a.slice, a.V);
  constexpr int E = Elt<T>::kPerGroup;
  c.ngroups = a.slice / E;

  T* data = reinterpret_cast<T*>(dsm);
  const size_t data_bytes = (size_t)a.slice * sizeof(T);
  c.gmax = reinterpret_cast<float*>(dsm + data_bytes);
  uint8_t* uni = dsm + data_bytes + (((size_t)c.ngroups * 4 + 15) & ~(size_t)15);
  c.gather = reinterpret_cast<uint64_t*>(uni);
  c.hmass = reinterpret_cast<unsigned long long*>(uni);
  c.hcnt = reinterpret_cast<unsigned int*>(uni + kBins * 8);
  c.mmass = reinterpret_cast<unsigned long long*>(uni + kBins * 12);
  c.mcnt = reinterpret_cast<unsigned int*>(uni + kBins * 12 + (size_t)(kBins / c.C) * 8);

  const RowParams P = a.params[c.row];
  c.greedy = (P.flags & kRowGreedy) != 0;
  c.inv_t = P.inv_t;
  c.ax = P.inv_t * kLog2e;
  c.top_k = P.top_k;
  c.top_p = P.top_p;
  c.topk = !c.greedy && P.top_k > 1 && P.top_k < a.V;
  c.topp = !c.greedy && (P.flags & kRowTopP) != 0;
  c.minp = !c.greedy && (P.flags & kRowMinP) != 0;
  c.lmp = P.log_min_p;
  c.rkey = row_key(a.seeds[c.row], c.row);
  const int n = a.n_logprobs;
  const int hist_len = a.hist_len[c.row];
  const bool pen = (P.flags & kRowPenalty) != 0 && hist_len > 0;
  c.tab = a.hist + (int64_t)c.row * a.hist_cap;
  c.zs = a.zside + (int64_t)c.row * a.hist_cap;
  c.e_lo = c.e_hi = 0;

  // ---- phase 0: stage the slice in shared memory ---------------------------
  const T* rowp = reinterpret_cast<const T*>(a.logits) + (int64_t)c.row * a.ld;
  const int nloc = max(0, c.hi - c.lo);
  if (c.tid == 0) {
    s.part.err = 0;
    s.gcount = 0;
    if (a.use_bulk) {
      mbar_init(&s.mbar, 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  int bulk_elems = 0;
  if (a.use_bulk) {
    const uint32_t bulk_bytes = ((uint32_t)nloc * (uint32_t)sizeof(T)) & ~15u;
    bulk_elems = (int)(bulk_bytes / sizeof(T));
    if (c.tid == 0) {
      mbar_arrive_expect_tx(&s.mbar, bulk_bytes);
      const char* src = reinterpret_cast<const char*>(rowp + c.lo);
      char* dst = reinterpret_cast<char*>(data);
      for (uint32_t off = 0; off < bulk_bytes; off += kBulkChunk)
        bulk_copy_g2s(dst + off, src + off, min(kBulkChunk, bulk_bytes - off), &s.mbar);
    }
  }
  for (int e = bulk_elems + c.tid; e < a.slice; e += kThreads) {
    if (e < nloc)
      Elt<T>::copy_global(data, e, rowp, (int64_t)c.lo + e);
    else
      Elt<T>::fill_neg_inf(data, e);
  }
  bool timed_out = false;
  if (a.use_bulk) timed_out = !mbar_wait_bounded(&s.mbar, 0);
  if (timed_out) {
    atomicOr(&s.part.err, kErrTimeout);
    mbar_wait_bounded(&s.mbar, 0);  // second bounded wait for the copy in flight
  }
  __syncthreads();

  // ---- phase 1: occurrence penalties into the side list ----------------------
  if (pen) {
    int below_lo = 0, below_hi = 0;
    for (int e = c.tid; e < hist_len; e += kThreads) {
      const int id = c.tab[e].x;
      below_lo += id < c.lo;
      below_hi += id < c.hi;
    }
    c.e_lo = block_sum_int(below_lo, s);
    c.e_hi = block_sum_int(below_hi, s);
    float* zs = a.zside + (int64_t)c.row * a.hist_cap;
    for (int e = c.e_lo + c.tid; e < c.e_hi; e += kThreads) {
      const int2 t = c.tab[e];
      const int local = t.x - c.lo;
      if (local < 0 || local >= nloc) {  // unsorted table: never write outside the slice
        atomicOr(&s.part.err, kErrInternal);
        continue;
      }
      zs[e] = penalize(Elt<T>::at(data, local), t.y, P);
      Elt<T>::mask(data, local);
    }
    __syncthreads();
  }

  // ---- phase 2: pass A (max, sum exp, argmax, group and thread maxima) -----
  {
    float rm = -INFINITY, rsum = 0.f, bv = -INFINITY;
    int bi = INT_MAX;
    bool nonfin = false;
    for (int g = c.tid; g < c.ngroups; g += kThreads) {
      float x[E];
      Elt<T>::load(data, g, x);
      float gm = x[0];
      bool nan = x[0] != x[0];
#pragma unroll
      for (int i = 1; i < E; ++i) {
        gm = fmaxf(gm, x[i]);
        nan |= x[i] != x[i];
      }
      nonfin |= nan;
      c.gmax[g] = gm;
      if (gm > rm) {
        rsum = (rm == -INFINITY) ? 0.f : rsum * ex2_approx((rm - gm) * c.ax);
        rm = gm;
      }
      if (rm > -INFINITY) {
        const float nb = -rm * c.ax;
        float e[E];
#pragma unroll
        for (int i = 0; i < E; ++i) e[i] = ex2_approx(fmaf(x[i], c.ax, nb));
#pragma unroll
        for (int w = 1; w < E; w <<= 1)
#pragma unroll
          for (int i = 0; i + w < E; i += 2 * w) e[i] += e[i + w];
        rsum += e[0];
      }
      if (gm > bv) {
        int first = 0;
#pragma unroll
        for (int i = E - 1; i >= 0; --i)
          if (x[i] == gm) first = i;
        bv = gm;
        bi = c.lo + g * E + first;
      }
    }
    for (int e = c.e_lo + c.tid; e < c.e_hi; e += kThreads) {
      const float z = c.zs[e];
      const int id = c.tab[e].x;
      nonfin |= z != z;
      if (z > rm) {
        rsum = (rm == -INFINITY) ? 0.f : rsum * ex2_approx((rm - z) * c.ax);
        rm = z;
      }
      if (rm > -INFINITY) rsum += ex2_approx(fmaf(z, c.ax, -rm * c.ax));
      if (pair_better(z, id, bv, bi)) {
        bv = z;
        bi = id;
      }
    }
    nonfin |= rm == INFINITY;
    s.tmax[c.tid] = rm;
    // CTA reduction
    float m = rm, sm = rsum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
      lse_combine(m, sm, m2, s2, c.ax);
    }
    float dz = 0.f;
    block_argmax(bv, bi, dz, s);
    const int nf = __syncthreads_or(nonfin);
    if (c.lane == 0) {
      s.rf[c.warp] = m;
      s.rf[kWarps + c.warp] = sm;
    }
    __syncthreads();
    if (c.tid == 0) {
      float mm = -INFINITY, ss = 0.f;
      for (int w = 0; w < kWarps; ++w) lse_combine(mm, ss, s.rf[w], s.rf[kWarps + w], c.ax);
      s.part.m = mm;
      s.part.s = ss;
      s.part.bv = bv;
      s.part.bi = bi;
      s.part.nonfinite = nf;
    }
  }
  cluster.sync();  // (1) pass-A partials visible
  if (c.warp == 0) {
    float m = -INFINITY, sm = 0.f, bv = -INFINITY;
    int bi = INT_MAX, nf = 0, er = 0;
    if (c.lane < c.C) {
      const Part* p = cluster.map_shared_rank(&s.part, c.lane);
      m = p->m;
      sm = p->s;
      bv = p->bv;
      bi = p->bi;
      nf = p->nonfinite;
      er = p->err;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
      lse_combine(m, sm, m2, s2, c.ax);
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (pair_better(v2, i2, bv, bi)) {
        bv = v2;
        bi = i2;
      }
      nf |= __shfl_xor_sync(0xffffffffu, nf, o);
      er |= __shfl_xor_sync(0xffffffffu, er, o);
    }
    if (c.lane == 0) {
      s.rs.M = m;
      s.rs.S = sm;
      s.rs.m_t = m * c.inv_t;
      s.rs.lnS = logf(sm);
      s.rs.bv = bv;
      s.rs.bi = bi;
      s.rs.nonfinite = nf || m == INFINITY || (m * c.inv_t) == INFINITY;
      s.rs.err = er;
    }
  }
  __syncthreads();
  c.m_t = s.rs.m_t;
  c.lnS = s.rs.lnS;
  const int status0 = s.rs.nonfinite ? kRowNonfinite : (s.rs.M == -INFINITY ? kRowEmpty : kRowOk);
  // Pass A sums 2^(x*log2e/T - max*log2e/T) with one FFMA per element; the
  // rounding of max*log2e/T makes that inexact once |max| is large.  Such rows
  // re-sum exp(z_t - m_t) from the tempered values themselves.
  if (status0 == kRowOk && fabsf(c.m_t) > 32.0f) {
    float acc = 0.f;
    for_each_elem<T>(
        c, data, [](float) { return true; },
        [&](float zt, int, bool) { acc += ex2_approx((zt - c.m_t) * kLog2e); });
    acc = block_sum_f(acc, s);
    if (c.tid == 0) s.part.s_exact = acc;
    cluster.sync();
    if (c.tid == 0) {
      float t = 0.f;
      for (int r = 0; r < c.C; ++r) t += cluster.map_shared_rank(&s.part, r)->s_exact;
      s.rs.S = t;
      s.rs.lnS = logf(t);
    }
    __syncthreads();
    c.lnS = s.rs.lnS;
  }
  const bool leader = c.rank == 0;
  int32_t* out_ids = n > 0 ? a.out_topk_ids + (int64_t)c.row * n : nullptr;
  float* out_lps = n > 0 ? a.out_topk_logprobs + (int64_t)c.row * n : nullptr;

  if (status0 != kRowOk) {
    cluster.sync();  // (2) nobody reads another CTA's shared memory after this
    if (leader) {
      if (c.tid < n) {
        out_ids[c.tid] = -1;
        out_lps[c.tid] = __int_as_float(0x7fc00000);
      }
      if (c.tid == 0) {
        a.out_tokens[c.row] = -1;
        if (a.out_logprobs) a.out_logprobs[c.row] = __int_as_float(0x7fc00000);
        a.row_status[c.row] = status0;
        a.dbg_kth_value[c.row] = __int_as_float(0x7fc00000);
        a.dbg_kth_index[c.row] = -1;
        a.dbg_kept[c.row] = 0;
        a.seeds[c.row] += kSeedStep;
        if (s.rs.err) atomicOr(a.err_word, s.rs.err);
      }
    }
    return;
  }

  // ---- phase 3: candidate threshold --------------------------------------
  int K_need = c.greedy ? n : max(n, c.topk ? c.top_k : ((c.topp || c.minp) ? kDefaultCand : 0));
  if (!c.greedy && !c.topk && (c.topp || c.minp)) K_need = min(K_need, max(n, c.C * kThreads));
  bool topk_beyond = false;
  if (K_need > c.C * kThreads) {
    K_need = n;
    topk_beyond = true;
  }
  float tau = INFINITY;
  if (K_need > 0) {
    const int Kc = (K_need + c.C - 1) / c.C;
    __syncthreads();
    bitonic_desc_f32(s.tmax, kThreads);
    if (c.tid == 0) s.part.tau = s.tmax[Kc - 1];
  }
  cluster.sync();  // (2) taus visible; pass-A partials no longer read
  if (K_need > 0) {
    if (c.warp == 0) {
      float t = INFINITY;
      if (c.lane < c.C) t = cluster.map_shared_rank(&s.part, c.lane)->tau;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t = fminf(t, __shfl_xor_sync(0xffffffffu, t, o));
      if (c.lane == 0) s.rs.tau = t;
    }
    __syncthreads();
    tau = s.rs.tau;
  }
  const bool complete = tau == -INFINITY;

  // ---- phase 4: pass B, candidates into the leader ---------------------------
  {
    int my_n = 0, my_minp = 0;
    unsigned long long my_mass = 0;
    if (K_need > 0) {
      const float tau_t = tau * c.inv_t;
      uint64_t* lg = cluster.map_shared_rank(c.gather, 0);
      int* lcount = cluster.map_shared_rank(&s.gcount, 0);
      for_each_elem<T>(
          c, data, [&](float gz) { return gz >= tau_t; },
          [&](float zt, int j, bool) {
            if (zt >= tau_t && zt > -INFINITY) {
              const int pos = atomicAdd(lcount, 1);
              if (pos < kGatherCap) lg[pos] = elem_key(zt, (uint32_t)j);
              ++my_n;
              my_mass += mass_fixed(zt, c.m_t);
              if (c.minp && minp_pass(zt, c.m_t, c.lmp)) ++my_minp;
            }
          });
    }
    my_n = block_sum_int(my_n, s);
    my_minp = block_sum_int(my_minp, s);
    my_mass = block_sum_u64(my_mass, s);
    if (c.tid == 0) {
      s.part.ncand = my_n;
      s.part.ncand_minp = my_minp;
      s.part.cand_mass = my_mass;
    }
  }
  cluster.sync();  // (3) candidates and their counts visible
  if (c.warp == 0) {
    int nc = 0, nm = 0;
    unsigned long long mass = 0;
    if (c.lane < c.C) {
      const Part* p = cluster.map_shared_rank(&s.part, c.lane);
      nc = p->ncand;
      nm = p->ncand_minp;
      mass = p->cand_mass;
    }
    nc = warp_sum_i(nc);
    nm = warp_sum_i(nm);
    mass = warp_sum_u64(mass);
    if (c.lane == 0) {
      s.rs.nc = nc;
      s.rs.nc_minp = nm;
      s.rs.cand_mass = mass;
    }
  }
  __syncthreads();
  const int nc = s.rs.nc;
  const bool cand_ok = K_need > 0 ? nc <= kGatherCap : true;
  const bool topn_ok = n == 0 || (cand_ok && nc >= n);
  const double S_fixed = (double)s.rs.S * 1099511627776.0;  // 2^40
  // The kept prefix is known from the candidates when every min-p survivor is
  // a candidate, or when top-k ends inside them; a top-p-only row also stays
  // fast when the candidates already hold more than p of the row's mass.
  const bool surv_inside = complete || (c.minp && s.rs.nc_minp < nc);
  const bool L2_inside = surv_inside || (c.topk && !topk_beyond && c.top_k <= nc);
  bool fast;
  if (c.greedy) {
    fast = topn_ok;
  } else {
    if (!c.topk && !c.topp && !c.minp)
      fast = complete && cand_ok;
    else if (c.topp)
      fast = cand_ok && (L2_inside || (!c.minp && !c.topk &&
                                       (double)s.rs.cand_mass >
                                           (double)c.top_p * S_fixed * (1.0 + 1e-5)));
    else
      fast = cand_ok && L2_inside;
    fast = fast && topn_ok && K_need > 0;
  }
  cluster.sync();  // (4) partials read; after this the fast path needs only the leader

  if (fast) {
    if (!leader) return;
    const int N = nc;
    const int P2 = pow2_ceil(max(N, 1));
    for (int i = N + c.tid; i < P2; i += kThreads) c.gather[i] = 0ull;
    __syncthreads();
    bitonic_desc_u64(c.gather, P2);
    for (int t = c.tid; t < n; t += kThreads) {
      const uint64_t k = c.gather[t];
      out_ids[t] = (int)key_idx(k);
      out_lps[t] = (key_z(k) - c.m_t) - c.lnS;
    }
    int tok;
    float ztok;
    int L3;
    if (c.greedy) {
      tok = s.rs.bi;
      ztok = c.m_t;
      L3 = 1;
    } else {
      // min-p prefix length among the candidates
      int pass = 0;
      if (c.minp)
        for (int i = c.tid; i < N; i += kThreads) pass += minp_pass(key_z(c.gather[i]), c.m_t, c.lmp);
      const int L1 = c.minp ? block_sum_int(pass, s) : N;
      const int L2 = c.topk ? min(c.top_k, L1) : L1;
      L3 = L2;
      if (c.topp) {
        const int per = (L2 + kThreads - 1) / kThreads;
        const int i0 = c.tid * per, i1 = min(L2, i0 + per);
        unsigned long long lm = 0;
        for (int i = i0; i < i1; ++i) lm += mass_fixed(key_z(c.gather[i]), c.m_t);
        unsigned long long tot;
        const unsigned long long ex = block_exclusive_u64(lm, s, &tot);
        const unsigned long long W2 = L2_inside ? tot : (unsigned long long)S_fixed;
        const unsigned long long Tm = (unsigned long long)((double)W2 * (double)c.top_p);
        int kept = 0;
        unsigned long long run = ex;
        for (int i = i0; i < i1; ++i) {
          if (run <= Tm) ++kept;
          run += mass_fixed(key_z(c.gather[i]), c.m_t);
        }
        L3 = max(1, block_sum_int(kept, s));
      }
      // Gumbel-max draw over the kept prefix
      float bs = -INFINITY, bz = 0.f;
      int bidx = INT_MAX;
      for (int i = c.tid; i < L3; i += kThreads) {
        const uint64_t k = c.gather[i];
        const int j = (int)key_idx(k);
        const float zt = key_z(k);
        const float sc = gumbel_score(zt, noise_bits(c.rkey, j));
        if (pair_better(sc, j, bs, bidx)) {
          bs = sc;
          bidx = j;
          bz = zt;
        }
      }
      block_argmax(bs, bidx, bz, s);
      tok = bidx;
      ztok = bz;
    }
    if (c.tid == 0) {
      const uint64_t kk = c.gather[L3 - 1];
      a.out_tokens[c.row] = tok;
      if (a.out_logprobs) a.out_logprobs[c.row] = (ztok - c.m_t) - c.lnS;
      a.row_status[c.row] = kRowOk;
      a.dbg_kth_value[c.row] = c.greedy ? c.m_t : key_z(kk);
      a.dbg_kth_index[c.row] = c.greedy ? tok : (int)key_idx(kk);
      a.dbg_kept[c.row] = L3;
      a.seeds[c.row] += kSeedStep;
      if (s.rs.err) atomicOr(a.err_word, s.rs.err);
    }
    if (a.update_counts) {
      __syncthreads();
      append_token(a.hist + (int64_t)c.row * a.hist_cap, a.hist_len + c.row, a.hist_cap, tok, s,
                   a.row_status + c.row);
    }
    return;
  }

  // ---- slow path: every CTA stays ------------------------------------------
  // top-n log-probs first (the gather buffer is reused below)
  if (n > 0) {
    if (topn_ok) {
      if (leader) {
        const int N = nc;
        const int P2 = pow2_ceil(max(N, 1));
        for (int i = N + c.tid; i < P2; i += kThreads) c.gather[i] = 0ull;
        __syncthreads();
        bitonic_desc_u64(c.gather, P2);
        for (int t = c.tid; t < n; t += kThreads) {
          const uint64_t k = c.gather[t];
          out_ids[t] = (int)key_idx(k);
          out_lps[t] = (key_z(k) - c.m_t) - c.lnS;
        }
      }
    } else {
      // rank n-1 of every non-NaN element (the -inf ones included, by index)
      SelOut so = cluster_select<T>(c, data, s, cluster, kPredAll, 0ull, false,
                                    (unsigned long long)(n - 1), 0.f);
      const unsigned long long kb = so.all ? 0ull : so.kb;
      if (leader && c.tid == 0) s.gcount = 0;
      cluster.sync();
      uint64_t* lg = cluster.map_shared_rank(c.gather, 0);
      int* lcount = cluster.map_shared_rank(&s.gcount, 0);
      const uint32_t kb_hi = (uint32_t)(kb >> 32);
      for_each_elem<T>(
          c, data, [&](float gz) { return ord_key(gz) >= kb_hi; },
          [&](float zt, int j, bool side) {
            if (j >= c.V) return;
            if (zt == -INFINITY && !side && is_side_slot(c, j)) return;
            const unsigned long long K = elem_key(zt, (uint32_t)j);
            if (K < kb) return;
            const int pos = atomicAdd(lcount, 1);
            if (pos < kGatherCap) lg[pos] = K;
          });
      cluster.sync();
      if (leader) {
        const int N = min(s.gcount, kGatherCap);
        const int P2 = pow2_ceil(max(N, 1));
        for (int i = N + c.tid; i < P2; i += kThreads) c.gather[i] = 0ull;
        __syncthreads();
        bitonic_desc_u64(c.gather, P2);
        for (int t = c.tid; t < n; t += kThreads) {
          if (t < N) {
            const uint64_t k = c.gather[t];
            out_ids[t] = (int)key_idx(k);
            out_lps[t] = (key_z(k) - c.m_t) - c.lnS;
          } else {
            out_ids[t] = -1;
            out_lps[t] = -INFINITY;
          }
        }
      }
    }
    cluster.sync();
  }

  int tok = -1;
  float ztok = 0.f;
  int kept = 1;
  float kth_v = c.m_t;
  int kth_i = s.rs.bi;
  if (c.greedy) {
    tok = s.rs.bi;
    ztok = c.m_t;
  } else {
    // kept set: threshold rows (no top-k, no top-p) or a selected boundary
    bool bounded = false;
    unsigned long long kb = 0ull;
    if (c.topk || c.topp) {
      unsigned long long kbk = 0ull;
      if (c.topk) {
        SelOut so = cluster_select<T>(c, data, s, cluster, kPredSurv, 0ull, false,
                                      (unsigned long long)(c.top_k - 1), 0.f);
        if (!so.all) {
          kbk = so.kb;
          bounded = true;
          kb = so.kb;
          kept = (int)so.cnt_incl;
        } else {
          kept = (int)so.total_cnt;
        }
      }
      if (c.topp) {
        SelOut so = cluster_select<T>(c, data, s, cluster, kPredSurv, kbk, true, 0ull, c.top_p);
        if (!so.all) {
          bounded = true;
          kb = so.kb;
          kept = (int)so.cnt_incl;
        } else {
          kept = (int)so.total_cnt;
        }
      }
    }
    // draw pass over the kept elements
    float s_cur = -INFINITY, bz = 0.f;
    int bidx = INT_MAX;
    int cnt = 0;
    unsigned long long kmin = ~0ull;
    const uint32_t kb_hi = (uint32_t)(kb >> 32);
    const bool threshold_row = !bounded;  // kept = every survivor: count it here
    for_each_elem<T>(
        c, data,
        [&](float gz) { return gz > -INFINITY && (!bounded || ord_key(gz) >= kb_hi); },
        [&](float zt, int j, bool) {
          if (!(zt > -INFINITY)) return;
          if (c.minp && !minp_pass(zt, c.m_t, c.lmp)) return;
          const unsigned long long K = elem_key(zt, (uint32_t)j);
          if (bounded && K < kb) return;
          if (threshold_row) {
            ++cnt;
            kmin = K < kmin ? K : kmin;
          }
          const uint32_t b = noise_bits(c.rkey, j);
          if (!may_beat(zt, s_cur, b)) return;
          const float sc = gumbel_score(zt, b);
          if (pair_better(sc, j, s_cur, bidx)) {
            s_cur = sc;
            bidx = j;
            bz = zt;
          }
        });
    block_argmax(s_cur, bidx, bz, s);
    cnt = block_sum_int(cnt, s);
    kmin = block_min_u64(kmin, s);
    if (c.tid == 0) {
      s.part.dscore = s_cur;
      s.part.didx = bidx;
      s.part.dz = bz;
      s.part.kept = cnt;
      s.part.kmin = kmin;
    }
    cluster.sync();
    if (leader && c.warp == 0) {
      float v = -INFINITY, z = 0.f;
      int i = INT_MAX, k2 = 0;
      unsigned long long km = ~0ull;
      if (c.lane < c.C) {
        const Part* p = cluster.map_shared_rank(&s.part, c.lane);
        v = p->dscore;
        i = p->didx;
        z = p->dz;
        k2 = p->kept;
        km = p->kmin;
      }
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
        k2 += __shfl_xor_sync(0xffffffffu, k2, o);
        const unsigned long long km2 = __shfl_xor_sync(0xffffffffu, km, o);
        km = km2 < km ? km2 : km;
      }
      if (c.lane == 0) {
        s.bcast_i[0] = i;
        s.bcast_f[0] = z;
        s.bcast_i[1] = k2;
        s.bcast_u[1] = km;
      }
    }
    cluster.sync();  // final: no DSMEM access after this
    if (!leader) return;
    __syncthreads();
    tok = s.bcast_i[0];
    ztok = s.bcast_f[0];
    if (threshold_row) {
      kept = s.bcast_i[1];
      kth_v = key_z(s.bcast_u[1]);
      kth_i = (int)key_idx(s.bcast_u[1]);
    } else {
      kth_v = key_z(kb);
      kth_i = (int)key_idx(kb);
    }
  }
  if (c.greedy) {
    cluster.sync();
    if (!leader) return;
  }
  if (c.tid == 0) {
    a.out_tokens[c.row] = tok;
    if (a.out_logprobs) a.out_logprobs[c.row] = (ztok - c.m_t) - c.lnS;
    a.row_status[c.row] = kRowOk;
    a.dbg_kth_value[c.row] = kth_v;
    a.dbg_kth_index[c.row] = kth_i;
    a.dbg_kept[c.row] = kept;
    a.seeds[c.row] += kSeedStep;
    const int er = s.rs.err | s.part.err;
    if (er) atomicOr(a.err_word, er);
  }
  if (a.update_counts) {
    __syncthreads();
    append_token(a.hist + (int64_t)c.row * a.hist_cap, a.hist_len + c.row, a.hist_cap, tok, s,
                 a.row_status + c.row);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side: plans and launches
// ---------------------------------------------------------------------------
static size_t union_bytes(int C) {
  const size_t hist = (size_t)kBins * 12 + (size_t)(kBins / C) * 12;
  const size_t gath = (size_t)kGatherCap * 8;
  return hist > gath ? hist : gath;
}

LaunchPlan plan_sample(int V, int elem_size) {
  // Smallest power-of-two cluster whose slices fit a ~48 KB staging budget
  // (several CTAs per SM), capped at 16 CTAs per row.
  const size_t target = 48 * 1024;
  int C = 1;
  while (C < kMaxCluster && (size_t)((V + C - 1) / C) * elem_size > target) C <<= 1;
  int slice = (V + C - 1) / C;
  slice = (slice + 15) & ~15;
  LaunchPlan p;
  p.cluster = C;
  p.slice = slice;
  const int E = kGroupBytes / elem_size;
  const size_t ngroups = (size_t)slice / E;
  p.smem = (size_t)slice * elem_size + ((ngroups * 4 + 15) & ~(size_t)15) + union_bytes(C);
  return p;
}

template <typename T>
static cudaError_t prepare_one(const LaunchPlan& plan, int* max_active) {
  cudaError_t e = cudaFuncSetAttribute(sample_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)plan.smem);
  if (e != cudaSuccess) return e;
  if (plan.cluster > 8) {
    e = cudaFuncSetAttribute(sample_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, sample_kernel<T>, &cfg);
  if (e != cudaSuccess) return e;
  if (max_active) *max_active = n;
  return n > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t prepare_sample(const LaunchPlan& plan, int dtype, int* max_active_clusters) {
  return dtype == 0 ? prepare_one<float>(plan, max_active_clusters)
                    : prepare_one<uint16_t>(plan, max_active_clusters);
}

template <typename T>
static cudaError_t launch_one(const SampleArgs& args, const LaunchPlan& plan,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)args.B * plan.cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_kernel<T>, args);
}

cudaError_t launch_sample(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                          cudaStream_t stream) {
  return dtype == 0 ? launch_one<float>(args, plan, stream)
                    : launch_one<uint16_t>(args, plan, stream);
}

}  // namespace vt
