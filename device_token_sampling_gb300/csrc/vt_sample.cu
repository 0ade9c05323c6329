// vt_sample.cu -- the fused batched decode sampling kernel for sm_103a.
//
// One thread-block cluster per logits row; each CTA owns a contiguous slice
// of the row.  The cluster size is chosen per call so that every row of the
// batch is resident at once (one wave): a row's latency then overlaps every
// other row's HBM stream, and HBM sees each logit once.
//
// Pipeline per row (pages: TensorRT-LLM "Sampling" for the penalty, temperature
// and filter formulas; vllm.cpp's Gumbel-draw pull request for the seeded
// draw and the lowest-index ArgReduce; the Tenstorrent sampling README for the
// log-softmax and the reset-then-sample state):
//   setup    the row's (id, count) entries inside the slice are penalised
//            (repetition, frequency, presence) into a side list, and a bitmap
//            marks their positions; every load of the slice patches them in
//            registers, so all passes see the penalised values;
//   pass A   16-byte vector loads stream the slice once: row max, sum of
//            exp (temperature folded into one FFMA), lowest-index argmax, a
//            conservative max per 32-byte group, and per-thread maxima, from
//            which each CTA derives a candidate threshold that admits at
//            least K/C of its elements (published with the pass-A partials);
//   pass B   only groups whose max clears the cluster-wide threshold are
//            re-read (from L2) and their candidates kept in shared memory;
//   leader   the candidates (a prefix of the order value desc, index asc) are
//            gathered into one CTA, sorted in registers, and min-p, top-k,
//            top-p and the Gumbel-max draw run on them;
//   slow     when the kept set reaches past the candidates (a wide top-p
//            nucleus, a large top-k, an unfiltered draw), a cluster-wide radix
//            select on 64-bit (value, index) keys with count/mass histograms
//            finds the exact boundary and a draw pass scores only elements
//            that can still win.
// Cross-CTA results move through distributed shared memory between hardware
// cluster barriers; no CTA spins on another.
#include "vt_device.cuh"
#include "vt_kernels.h"

#include <climits>

namespace cg = cooperative_groups;

namespace vt {
namespace {

constexpr int kBufCap = 2048;       // candidate keys a CTA (and the leader) can hold
constexpr int kBinBits = 10;
constexpr int kBins = 1 << kBinBits;
constexpr int kDefaultCand = 512;   // candidates tried for top-p / min-p rows
constexpr int kGroupBytes = 32;     // one thread step: two 16-byte vectors
constexpr int kMaxCluster = 16;
constexpr int kGroupsPerStage = 2;                   // groups a thread consumes per stage
constexpr int kStageBytes = kThreads * kGroupBytes * kGroupsPerStage;  // 16 KB a stage
constexpr int kStages = 2;                           // bulk-copy ring depth of pass A
constexpr int kRingBytes = kStageBytes * kStages;    // aliases the candidate buffer
constexpr int kSmallK = 32;  // up to this many per CTA, thresholds come from thread maxima
constexpr int kSideSmem = 2048;  // penalised values of a slice held in shared memory
// the ring region also holds the candidate buffer (kBufCap keys) followed by
// the level-0 per-bin bests; the histograms alias the buffer
static_assert(kBufCap * 8 <= kRingBytes, "the candidate buffer lives in the ring region");
static_assert((1 << 10) * 16 <= kBufCap * 8, "selection histograms exceed the gather buffer");

template <typename T>
struct Elt;

template <>
struct Elt<float> {
  static constexpr int E = kGroupBytes / 4;
  __device__ static void load_vec(const float* p, float* x) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    const uint4 a = __ldg(q), b = __ldg(q + 1);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  }
  __device__ static float load1(const float* p) { return __ldg(p); }
  __device__ static void unpack(const uint4& a, const uint4& b, float* x) {
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  }
};

// bfloat16 stored as its 16 bits; widening to fp32 is exact (a 16-bit shift).
template <>
struct Elt<uint16_t> {
  static constexpr int E = kGroupBytes / 2;
  __device__ static void load_vec(const uint16_t* p, float* x) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    const uint4 a = __ldg(q), b = __ldg(q + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static float load1(const uint16_t* p) {
    return __uint_as_float((uint32_t)__ldg(p) << 16);
  }
  __device__ static void unpack(const uint4& a, const uint4& b, float* x) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

// Group maxima are kept as the largest bf16 value <= the true maximum: a lower
// bound for the candidate threshold, and (one bf16 step up) an upper bound for
// the group filters, so both stay exact.
__device__ __forceinline__ uint16_t bf16_down(float f) {
  const uint32_t u = __float_as_uint(f);
  if (f != f) return 0x7FC0u;
  if (u & 0x80000000u) return (uint16_t)((u >> 16) + ((u & 0xFFFFu) ? 1u : 0u));
  return (uint16_t)(u >> 16);
}
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// The next bf16 value above b (an upper bound of the group's true maximum).
__device__ __forceinline__ float bf16_next_up(uint16_t b) {
  uint32_t n;
  if (b == 0xFF80u) return -INFINITY;  // a group of -inf stays -inf
  if (b & 0x8000u)
    n = (b & 0x7FFFu) ? (uint32_t)(b - 1u) : 0x0001u;
  else
    n = (b >= 0x7F80u) ? b : (uint32_t)(b + 1u);
  return __uint_as_float(n << 16);
}
// Per-CTA partial results; other CTAs of the cluster read them over DSMEM.
struct Part {
  float m, s, bv;
  int bi;
  int nonfinite;
  float tau, tau_n;  // candidate thresholds: for the kept set, for top-n only
  int ncand, ncand_minp;
  unsigned long long cand_mass;
  unsigned long long rng_cnt, rng_mass;
  unsigned long long rng_all, rng_tmass;  // code walk: range totals
  int rng_last;
  float best_score;      // code walk: best wholly kept slot of the range
  int best_slot, best_tie;
  unsigned int best_bits;
  float dscore, dz;
  int didx;
  int kept;
  unsigned long long kmin;
  unsigned long long tiny_mass, catch_mass;  // code bins: masses summed per element
  // selection on bf16 codes: the two several-valued slots (tiny, catch-all)
  unsigned long long sp_all[2], sp_cnt[2], sp_mass[2];
  unsigned long long sp_key[2];  // best (Gumbel score, index) key of each
  unsigned long long cb_key;     // best ((bits + 1), ~index) in the boundary slot's kept prefix
  int cb_last;           // the last kept index of the boundary slot
  int cw_j;              // lowest index of the winning slot's best element
  int last_j;            // last index of the last survivor slot (no boundary)
  int err;
};

// Outcome of the leader's walk over the bf16 code slots.
struct CodeWalk {
  int fallback;       // the row needs the generic selection
  int slot, kp;       // boundary slot and its kept elements (slot -1: all survivors kept)
  unsigned long long above;  // survivors before the boundary slot
  unsigned long long total;  // survivors
  int last_slot;      // last occupied survivor slot
  int nwin;           // 1 when a wholly kept regular slot holds the best score
  int wslot;          // that slot
  unsigned int wb;    // its best noise bits + 1
  float wscore;
  int sp_kept[2];     // the tiny / catch-all slot is wholly kept
  unsigned long long sp_all[2], sp_cnt[2], sp_mass[2], sp_key[2];  // their totals
  int slot_n, kn;     // top-n boundary slot and its elements in the top-n (-1: none)
  int k_slot, k_kept; // top-k boundary slot and its kept elements
  unsigned long long k_mass;  // mass of the top-k set
};

struct RowStats {
  float S, m_t, lnS, bv;
  int bi;
  int nonfinite;
  float tau, tau_n;
  int nc, nc_minp, push_off, overflow;
  unsigned long long cand_mass;
  int err;
};

struct SelOut {
  unsigned long long kb, cnt_incl, mass_incl, total_cnt, total_mass;
  unsigned long long win;  // best (score, index) key over the kept set when draw_ok
  int all;
  int draw_ok;
};

struct Walk {
  int d;
  int found;
  unsigned long long acc_c, acc_m, band_cnt, total_c, total_m;
};

struct __align__(16) Smem {
  uint64_t full[kStages];  // bulk-copy completion, one mbarrier per ring slot
  unsigned int hist256[256];
  Part part;
  RowStats rs;
  SelOut sel;
  Walk walk;
  CodeWalk cw;
  int nloc;    // candidates in this CTA's buffer
  int gcount;  // band keys gathered in the leader (selection)
  int gcount2;  // boundary-slot indices gathered in the leader (code selection)
  int bcast_i[4];
  float bcast_f[4];
  unsigned long long bcast_u[4];
  __align__(16) float tmax[kThreads];
  float rf[kWarps * 4];
  int ri[kWarps * 4];
  unsigned long long ru[kWarps * 4];
};

struct Ctx {
  int tid, lane, warp;
  int C, rank, row, V, lo, hi, slice, ngroups;
  bool aligned, pen;
  float inv_t, ax;  // 1/T and log2(e)/T
  float m_t, lnS;   // row max of z_t, ln(sum exp(z_t - m_t))
  float xmax;       // the row maximum before temperature (selection kernel)
  bool greedy, topk, topp, minp;
  int top_k;
  float top_p;
  double lmp;       // ln(min_p)
  const void* rowp;
  uint16_t* gmax;   // conservative bf16 max of each group (pre-temperature)
  uint64_t* buf;    // candidate keys / gathered keys / histograms
  unsigned int* hcnt;  // selection histogram: counts, then three partial mass sums
  unsigned int* mcnt;  // merged bins of this CTA's digit range
  unsigned long long* mmass;
  const uint32_t* bitmap;  // penalised positions of the slice
  const uint16_t* prefix;  // side-list index of each bitmap word's first bit
  const float* side_z;     // penalised values, in id order, of this slice
  const uint4* stage;      // the slice copied to shared memory (selection kernel), or null
  uint64_t rkey;           // noise stream key
  unsigned long long* trace;  // optional phase trace of this CTA (kTraceSlots stamps)
};

// Phase stamp from inside helpers (slot k of this CTA's trace).
#define VT_CTRACE(c, k)                                                   \
  do {                                                                    \
    if ((c).trace && threadIdx.x == 0) (c).trace[(k)] = global_timer_ns(); \
  } while (0)

// Optional phase trace: thread 0 stamps the global timer into slot k.
// Phase stamp of the streaming kernel (slot k of this CTA's trace, laid out
// by row and rank).
#define VT_TRACE(k) VT_CTRACE(c, k)

// ---------------------------------------------------------------------------
// loading one 32-byte group of the slice into registers
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void patch_group(const Ctx& c, int g, float* x);

template <typename T>
__device__ __forceinline__ void load_group(const Ctx& c, int g, float* x) {
  constexpr int E = Elt<T>::E;
  if (c.stage) {  // staged slices are padded with -inf to whole groups
    Elt<T>::unpack(c.stage[2 * g], c.stage[2 * g + 1], x);
    patch_group<T>(c, g, x);
    return;
  }
  const T* row = reinterpret_cast<const T*>(c.rowp);
  const int j0 = c.lo + g * E;
  if (c.aligned && j0 + E <= c.hi) {
    Elt<T>::load_vec(row + j0, x);
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = (j0 + i < c.hi) ? Elt<T>::load1(row + j0 + i) : -INFINITY;
  }
  patch_group<T>(c, g, x);
}

// Replace the penalised positions of group g by their side-list values.
template <typename T>
__device__ __forceinline__ void patch_group(const Ctx& c, int g, float* x) {
  constexpr int E = Elt<T>::E;
  if (c.pen) {
    const int bit0 = g * E;
    const uint32_t word = c.bitmap[bit0 >> 5];
    const uint32_t m = (word >> (bit0 & 31)) & ((E == 32) ? 0xFFFFFFFFu : ((1u << E) - 1u));
    if (m != 0u) {
      int idx = (int)c.prefix[bit0 >> 5] + __popc(word & ((1u << (bit0 & 31)) - 1u));
#pragma unroll
      for (int i = 0; i < E; ++i) {
        if (m & (1u << i)) {
          x[i] = c.side_z[idx];
          ++idx;
        }
      }
    }
  }
}

// Visit the elements of every group whose conservative max passes
// group_ok(max * inv_t); elem(zt, j) gets the tempered value and global index.
template <typename T, typename GF, typename FN>
__device__ __forceinline__ void for_each_group(const Ctx& c, GF group_ok, FN fn) {
  // Groups whose conservative max passes group_ok(max * inv_t), in the order
  // g = tid, tid + kThreads, ...; the next such group's 32 bytes are loaded
  // while the current one is processed.  fn(x, g, j0) gets the (penalised)
  // pre-temperature values of elements j0 .. j0 + E - 1 (-inf past the row).
  constexpr int E = Elt<T>::E;
  auto next_ok = [&](int g) {
    while (g < c.ngroups && !group_ok(__fmul_rn(bf16_next_up(c.gmax[g]), c.inv_t))) g += kThreads;
    return g;
  };
  auto vec_ok = [&](int g) {
    return c.stage != nullptr || (c.aligned && c.lo + (g + 1) * E <= c.hi);
  };
  auto fetch = [&](int g, uint4& u0, uint4& u1) {
    if (c.stage) {
      u0 = c.stage[2 * g];
      u1 = c.stage[2 * g + 1];
      return;
    }
    const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(c.rowp) + c.lo +
                                                    g * E);
    u0 = __ldg(q);
    u1 = __ldg(q + 1);
  };
  int g = next_ok(c.tid);
  uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
  if (g < c.ngroups && vec_ok(g)) fetch(g, a0, a1);
  while (g < c.ngroups) {
    const int gn = next_ok(g + kThreads);
    uint4 b0 = make_uint4(0, 0, 0, 0), b1 = b0;
    if (gn < c.ngroups && vec_ok(gn)) fetch(gn, b0, b1);
    float x[E];
    if (vec_ok(g)) {
      Elt<T>::unpack(a0, a1, x);
      patch_group<T>(c, g, x);
    } else {
      load_group<T>(c, g, x);
    }
    fn(x, g, c.lo + g * E);
    a0 = b0;
    a1 = b1;
    g = gn;
  }
}

// Elementwise view of for_each_group: elem(zt, j) gets the tempered value
// fl(x * (1/T)) and the global index of every element of the row.
template <typename T, typename GF, typename EF>
__device__ __forceinline__ void for_each_elem(const Ctx& c, GF group_ok, EF elem) {
  constexpr int E = Elt<T>::E;
  for_each_group<T>(c, group_ok, [&](float* x, int, int j0) {
#pragma unroll
    for (int i = 0; i < E; ++i)
      if (j0 + i < c.hi) elem(__fmul_rn(x[i], c.inv_t), j0 + i);
  });
}

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

__device__ unsigned long long block_max_u64(unsigned long long v, Smem& s) {
  return ~block_min_u64(~v, s);
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
    const unsigned long long t = threadIdx.x < kWarps ? s.ru[threadIdx.x] : 0ull;
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

// Descending bitonic sort of KPT * kThreads keys held KPT per thread
// (consecutive), exchanging through registers, warp shuffles, and shared
// memory only for partners in other warps.
template <int KPT>
__device__ void block_sort_desc_impl(uint64_t* keys) {
  constexpr int N = KPT * kThreads;
  uint64_t v[KPT];
  const int base = threadIdx.x * KPT;
#pragma unroll
  for (int q = 0; q < KPT; ++q) v[q] = keys[base + q];
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < KPT) {
        // partners within the thread: one unrolled case per distance, so that
        // every index into v is known at compile time (v stays in registers)
#pragma unroll
        for (int jj = KPT / 2; jj > 0; jj >>= 1) {
          if (jj == j) {
#pragma unroll
            for (int q = 0; q < KPT; ++q) {
              const int p = q ^ jj;
              if (p > q) {
                const bool up = ((base + q) & k) == 0;
                const uint64_t a = v[q], b = v[p];
                if (up ? (a < b) : (a > b)) {
                  v[q] = b;
                  v[p] = a;
                }
              }
            }
          }
        }
      } else if (j < 32 * KPT) {
        const int lm = j / KPT;
#pragma unroll
        for (int q = 0; q < KPT; ++q) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, v[q], lm);
          const int i = base + q;
          const bool lower = (i & j) == 0;
          const bool up = (i & k) == 0;
          v[q] = (lower == up) ? (v[q] > o ? v[q] : o) : (v[q] < o ? v[q] : o);
        }
      } else {
#pragma unroll
        for (int q = 0; q < KPT; ++q) keys[base + q] = v[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < KPT; ++q) {
          const int i = base + q;
          const uint64_t o = keys[i ^ j];
          const bool lower = (i & j) == 0;
          const bool up = (i & k) == 0;
          v[q] = (lower == up) ? (v[q] > o ? v[q] : o) : (v[q] < o ? v[q] : o);
        }
        __syncthreads();
      }
    }
  }
#pragma unroll
  for (int q = 0; q < KPT; ++q) keys[base + q] = v[q];
  __syncthreads();
}

// Sort keys[0, n) descending (n <= kBufCap); pads with zeros up to a power of
// two of at least kThreads.
__device__ void block_sort_desc(uint64_t* keys, int n) {
  int P2 = kThreads;
  while (P2 < n) P2 <<= 1;
  for (int i = n + threadIdx.x; i < P2; i += kThreads) keys[i] = 0ull;
  __syncthreads();
  if (P2 <= kThreads)
    block_sort_desc_impl<1>(keys);
  else if (P2 <= 2 * kThreads)
    block_sort_desc_impl<2>(keys);
  else if (P2 <= 4 * kThreads)
    block_sort_desc_impl<4>(keys);
  else
    block_sort_desc_impl<8>(keys);
}

// The K-th largest of N distinct keys (1 <= K <= N), most significant byte
// first: a 256-bin count of the keys that share the prefix found so far, the
// bin holding rank K, then the next byte.  Ends as soon as that bin holds one
// key.  All threads of the CTA call it and get the key.
__device__ uint64_t block_select_desc(const uint64_t* keys, int N, int K, Smem& s) {
  uint64_t prefix = 0ull, mask = 0ull;
  int need = K;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += kThreads) s.hist256[b] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += kThreads) {
      const uint64_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&s.hist256[(uint32_t)(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l takes bins 255 - 8l down to 248 - 8l: descending key order
      const int lane = threadIdx.x;
      unsigned int cnt[8], tot = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cnt[q] = s.hist256[255 - 8 * lane - q];
        tot += cnt[q];
      }
      unsigned int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int w = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += w;
      }
      const unsigned int excl = incl - tot;
      if (excl < (unsigned int)need && (unsigned int)need <= incl) {
        unsigned int run = excl;
        int bin = -1, nn = 0, bc = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (bin < 0 && run + cnt[q] >= (unsigned int)need) {
            bin = 255 - 8 * lane - q;
            nn = need - (int)run;
            bc = (int)cnt[q];
          }
          run += cnt[q];
        }
        s.bcast_i[0] = bin;
        s.bcast_i[1] = nn;
        s.bcast_i[2] = bc;
      }
    }
    __syncthreads();
    const int bin = s.bcast_i[0];
    need = s.bcast_i[1];
    const int bc = s.bcast_i[2];
    prefix |= (uint64_t)(uint32_t)bin << shift;
    mask |= 255ull << shift;
    __syncthreads();  // the broadcast is read before anyone writes it again
    if (bc == 1 || shift == 0) {
      for (int i = threadIdx.x; i < N; i += kThreads)
        if ((keys[i] & mask) == prefix) s.bcast_u[0] = keys[i];
      __syncthreads();
      const uint64_t r = s.bcast_u[0];
      __syncthreads();
      return r;
    }
  }
  return prefix;  // not reached: the last byte leaves one key
}

// Descending bitonic sort of keys[0, n), n <= 32, by one warp (keys past n
// read as 0, the smallest key).
__device__ __forceinline__ void warp_sort_desc32(uint64_t* keys, int n, int lane) {
  uint64_t v = lane < n ? keys[lane] : 0ull;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool lower = (lane & j) == 0;
      const bool up = (lane & k) == 0;
      v = (lower == up) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  if (lane < n) keys[lane] = v;
}

// The q largest of N distinct keys (q <= 32), sorted descending into out[0, q):
// a selection of the q-th, a gather of the keys at or above it, a warp sort.
__device__ void block_top_desc(const uint64_t* keys, int N, int q, uint64_t* out, Smem& s) {
  const uint64_t kq = block_select_desc(keys, N, q, s);
  if (threadIdx.x == 0) s.bcast_i[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += kThreads) {
    const uint64_t k = keys[i];
    if (k >= kq) out[atomicAdd(&s.bcast_i[3], 1)] = k;
  }
  __syncthreads();
  if (threadIdx.x < 32) warp_sort_desc32(out, q, threadIdx.x);
  __syncthreads();
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
//
// Level 0 bins by distance below the row max (1/64 per bin, the last bin
// catches everything from 16 down), which spreads any row's mass over many
// bins; deeper levels split the surviving bin's 64-bit key range 1024 ways.
// A band of at most kBufCap keys is then gathered, sorted and walked.  Bin
// masses are exact sums of the elements' 2^-43 fixed-point masses, kept as
// three 32-bit partial sums per bin so that every update is a 32-bit shared
// atomic (slices of at most 65536 elements cannot overflow them).
//
// With with_draw, the pass that gathers the band also draws over the
// elements above it (all kept): each thread keeps its best Gumbel score, and
// the leader combines those with the kept prefix of the sorted band.  The
// winner's key comes back in `win` (draw_ok).
constexpr float kDScale = 64.0f;
constexpr unsigned long long kNegInfKey = 0x007FFFFF00000000ull;  // elem_key(-inf, ~0)

// tempered value of regular slot sl below the maximum code cmax
__device__ __forceinline__ float zq_value(int cmax, int sl, float inv_t) {
  return __fmul_rn(code_value(cmax - sl), inv_t);
}

// Histogram words: count, then the three partial mass sums, kBins each.
__device__ __forceinline__ void hist_add(unsigned int* h, int d, unsigned long long q,
                                         bool by_mass) {
  atomicAdd(&h[d], 1u);
  if (by_mass) {
    atomicAdd(&h[kBins + d], (unsigned int)(q & 0xFFFFull));
    atomicAdd(&h[2 * kBins + d], (unsigned int)((q >> 16) & 0xFFFFull));
    atomicAdd(&h[3 * kBins + d], (unsigned int)(q >> 32));
  }
}
__device__ __forceinline__ unsigned long long hist_mass(const unsigned int* h, int d) {
  return (unsigned long long)h[kBins + d] + ((unsigned long long)h[2 * kBins + d] << 16) +
         ((unsigned long long)h[3 * kBins + d] << 32);
}

template <typename T>
__device__ __noinline__ SelOut cluster_select(Ctx& c, Smem& s, cg::cluster_group& cluster,
                                              int pred, unsigned long long kbound, bool by_mass,
                                              unsigned long long count_target, float p,
                                              bool with_draw, bool codes) {
  constexpr int E = Elt<T>::E;
  // values the scans use, in registers
  const float m_t = c.m_t, inv_t = c.inv_t;
  const int hi = c.hi;
  const bool minp = c.minp;
  const double lmp = c.lmp;
  const uint64_t rkey = c.rkey;
  unsigned int* const h = c.hcnt;
  unsigned long long Klo = kbound, Khi = ~0ull;
  unsigned long long acc_c = 0, acc_m = 0;
  unsigned long long target = count_target;
  unsigned long long total_c = 0, total_m = 0;
  int dsel = -1;  // the level-0 bin every later level stays inside
  SelOut out;
  out.all = 0;
  out.draw_ok = 0;
  out.win = kNegInfKey;
  const int nslots0 = codes ? kCodeSlots : kBins;  // level-0 bins
  const int cmax = codes ? code16(__float_as_uint(c.xmax) >> 16) : 0;
  const int tiny_slot = (cmax >= 0 && cmax < kCodeSlots - 1) ? cmax : -1;

  auto in_pred = [&](float zt) -> bool {
    if (pred == kPredAll) return true;
    if (!(zt > -INFINITY)) return false;
    return !minp || minp_pass(zt, m_t, lmp);
  };
  auto dbin = [&](float zt) -> int {
    const float d = __fsub_rn(m_t, zt) * kDScale;  // exact scaling of a rounded difference
    return d < (float)(kBins - 1) ? (int)d : kBins - 1;
  };
  // level-0 bin of an element (x before temperature, zt after)
  auto slot = [&](float x, float zt) -> int {
    if (!codes) return dbin(zt);
    const int d = cmax - code16(__float_as_uint(x) >> 16);
    return d < kCodeSlots - 1 ? d : kCodeSlots - 1;
  };
  // mass of the level-0 bin b holding n elements (code bins only)
  auto code_mass = [&](int b, unsigned long long n, unsigned long long tiny,
                       unsigned long long catchall) -> unsigned long long {
    if (b == tiny_slot) return tiny;
    if (b == kCodeSlots - 1) return catchall;
    if (n == 0) return 0ull;
    return n * mass_fixed(__fmul_rn(code_value(cmax - b), inv_t), m_t);
  };

  for (int level = 0; level < 8; ++level) {
    const bool dlevel = level == 0;
    const bool cl = dlevel && codes;  // this level bins by bf16 code
    const int nb = (dlevel ? nslots0 : kBins) / c.C, b0 = c.rank * nb;
    const unsigned long long range = Khi - Klo;
    const int bits = range == 0 ? 0 : 64 - __clzll((long long)range);
    const int shift = bits > kBinBits ? bits - kBinBits : 0;
    for (int b = c.tid; b < 4 * kBins; b += kThreads) h[b] = 0u;
    __syncthreads();
    if (dlevel) VT_CTRACE(c, 4);
    const uint32_t klo_hi = (uint32_t)(Klo >> 32);
    if (cl) {
      // one count per element; the masses of the two several-valued bins are
      // summed per element
      unsigned long long tm = 0ull, cm = 0ull;
      for_each_group<T>(
          c, [&](float gz) { return ord_key(gz) >= klo_hi; },
          [&](float* x, int, int j0) {
#pragma unroll
            for (int i = 0; i < E; ++i) {
              const float zt = __fmul_rn(x[i], inv_t);
              const int j = j0 + i;
              if (j >= hi || !in_pred(zt)) continue;
              if (kbound != 0ull && elem_key(zt, (uint32_t)j) < kbound) continue;
              const int d = slot(x[i], zt);
              atomicAdd(&h[d], 1u);
              if (by_mass) {
                if (d == tiny_slot) tm += mass_fixed(zt, m_t);
                if (d == kCodeSlots - 1) cm += mass_fixed(zt, m_t);
              }
            }
          });
      tm = block_sum_u64(tm, s);
      cm = block_sum_u64(cm, s);
      if (c.tid == 0) {
        s.part.tiny_mass = tm;
        s.part.catch_mass = cm;
      }
      VT_CTRACE(c, 12);
    } else if (dlevel) {
      // the catch-all bin is summed per thread (no contention on one word)
      unsigned int cc = 0u;
      unsigned long long cm = 0ull;
      for_each_group<T>(
          c, [&](float gz) { return ord_key(gz) >= klo_hi; },
          [&](float* x, int, int j0) {
#pragma unroll
            for (int i = 0; i < E; ++i) {
              const float zt = __fmul_rn(x[i], inv_t);
              const int j = j0 + i;
              if (j >= hi || !in_pred(zt)) continue;
              if (kbound != 0ull && elem_key(zt, (uint32_t)j) < kbound) continue;
              const int d = dbin(zt);
              const unsigned long long q = by_mass ? mass_fixed(zt, m_t) : 0ull;
              if (d == kBins - 1) {
                ++cc;
                cm += q;
              } else {
                hist_add(h, d, q, by_mass);
              }
            }
          });
      if (cc) {
        atomicAdd(&h[kBins - 1], cc);
        if (by_mass) {
          atomicAdd(&h[2 * kBins - 1], (unsigned int)(cm & 0xFFFFull));
          atomicAdd(&h[3 * kBins - 1], (unsigned int)((cm >> 16) & 0xFFFFull));
          atomicAdd(&h[4 * kBins - 1], (unsigned int)(cm >> 32));
        }
      }
      VT_CTRACE(c, 12);
    } else {
      const unsigned long long lo = Klo, hk = Khi;
      const int ds = dsel;
      for_each_group<T>(
          c, [&](float gz) { return ord_key(gz) >= klo_hi; },
          [&](float* x, int, int j0) {
#pragma unroll
            for (int i = 0; i < E; ++i) {
              const float zt = __fmul_rn(x[i], inv_t);
              const int j = j0 + i;
              if (j >= hi || !in_pred(zt)) continue;
              const unsigned long long K = elem_key(zt, (uint32_t)j);
              if (K < lo || K > hk || slot(x[i], zt) != ds) continue;
              hist_add(h, (int)((hk - K) >> shift), by_mass ? mass_fixed(zt, m_t) : 0ull,
                       by_mass);
            }
          });
    }
    cluster.sync();
    // distributed merge: this CTA sums its digit range over the cluster
    unsigned long long my_c = 0, my_m = 0;
    unsigned long long tiny_all = 0, catch_all = 0;
    if (cl && by_mass && c.tid < c.C) {
      const Part* pr = cluster.map_shared_rank(&s.part, c.tid);
      tiny_all = pr->tiny_mass;
      catch_all = pr->catch_mass;
    }
    if (cl && by_mass) {
      tiny_all = warp_sum_u64(c.lane < c.C ? tiny_all : 0ull);
      catch_all = warp_sum_u64(c.lane < c.C ? catch_all : 0ull);
      if (c.lane == 0 && c.warp == 0) {
        s.bcast_u[2] = tiny_all;
        s.bcast_u[3] = catch_all;
      }
      __syncthreads();
      tiny_all = s.bcast_u[2];
      catch_all = s.bcast_u[3];
    }
    for (int b = c.tid; b < nb; b += kThreads) {
      unsigned long long sc = 0, sm = 0;
      for (int r = 0; r < c.C; ++r) {
        const unsigned int* hr = cluster.map_shared_rank(h, r);
        sc += hr[b0 + b];
        if (by_mass && !cl) sm += hist_mass(hr, b0 + b);
      }
      if (by_mass && cl) sm = code_mass(b0 + b, sc, tiny_all, catch_all);
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
      if (dlevel && by_mass) tgt = (unsigned long long)((double)tm * (double)p);
      const unsigned long long base_c = acc_c, base_m = acc_m;
      const bool cross =
          c.lane < c.C && (by_mass ? (base_m + im > tgt) : (base_c + ic > tgt));
      const unsigned int mask = __ballot_sync(0xffffffffu, cross);
      if (c.lane == 0) {
        s.walk.found = mask != 0;
        s.bcast_u[0] = tgt;
      }
      if (mask != 0) {
        const int r = __ffs(mask) - 1;
        const unsigned long long before_c = base_c + __shfl_sync(0xffffffffu, ic - rc, r);
        const unsigned long long before_m = base_m + __shfl_sync(0xffffffffu, im - rm, r);
        const unsigned int* mc = cluster.map_shared_rank(c.mcnt, r);
        const unsigned long long* mm = cluster.map_shared_rank(c.mmass, r);
        unsigned long long run_c = before_c, run_m = before_m;
        int dpick = -1;
        unsigned long long sel_c = 0, sel_m = 0, band = 0;
        for (int base = 0; base < nb && dpick < 0; base += 32) {
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
            dpick = r * nb + base + l;
            sel_c = run_c + __shfl_sync(0xffffffffu, xc - vc, l);
            sel_m = run_m + __shfl_sync(0xffffffffu, xm - vm, l);
            band = __shfl_sync(0xffffffffu, vc, l);
          } else {
            run_c += __shfl_sync(0xffffffffu, xc, 31);
            run_m += __shfl_sync(0xffffffffu, xm, 31);
          }
        }
        if (c.lane == 0) {
          s.walk.d = dpick;
          s.walk.acc_c = sel_c;
          s.walk.acc_m = sel_m;
          s.walk.band_cnt = band;
        }
      }
    }
    __syncthreads();
    if (dlevel) {
      total_c = s.walk.total_c;
      total_m = s.walk.total_m;
      target = s.bcast_u[0];
    }
    const bool found = s.walk.found;
    const int d = s.walk.d;
    const unsigned long long band = s.walk.band_cnt;
    acc_c = s.walk.acc_c;
    acc_m = s.walk.acc_m;
    if (c.rank == 0 && c.tid == 0) s.gcount = 0;
    if (!found) {
      cluster.sync();  // merged arrays and parts are free again
      out.all = 1;
      out.kb = kbound;
      out.cnt_incl = total_c;
      out.mass_incl = total_m;
      out.total_cnt = total_c;
      out.total_mass = total_m;
      return out;
    }
    if (cl) {
      // the key range of code bin d: one value, or (code 0, catch-all) the
      // range of its values, widened so that rounding cannot leave it
      dsel = d;
      if (d != tiny_slot && d != kCodeSlots - 1) {
        const float zv = __fmul_rn(code_value(cmax - d), inv_t);
        Khi = elem_key(zv, 0u);
        const unsigned long long klo = elem_key(zv, 0xFFFFFFFFu);
        Klo = klo > kbound ? klo : kbound;
      } else {
        const float zh = (d == tiny_slot) ? __fmul_rn(0x1p-12f, inv_t)
                                          : __fmul_rn(code_value(cmax - (kCodeSlots - 2)), inv_t);
        const float margin = 1e-3f * (1.0f + fabsf(zh));
        Khi = elem_key(zh + margin, 0u);
        const unsigned long long klo =
            (d == tiny_slot) ? elem_key(-zh - margin, 0xFFFFFFFFu) : 0ull;
        Klo = klo > kbound ? klo : kbound;
      }
    } else if (dlevel) {
      // the key range of bin d, widened so that rounding cannot leave it
      dsel = d;
      const float margin = 1e-3f * (1.0f + fabsf(m_t));
      const float z_hi = m_t - (float)d / kDScale + margin;
      const float z_lo = (d == kBins - 1) ? -INFINITY : m_t - (float)(d + 1) / kDScale - margin;
      Khi = elem_key(z_hi, 0u);
      const unsigned long long klo = (d == kBins - 1) ? 0ull : elem_key(z_lo, 0xFFFFFFFFu);
      Klo = klo > kbound ? klo : kbound;
    } else {
      const unsigned long long hi_new = Khi - ((unsigned long long)d << shift);
      const unsigned long long width = (1ull << shift) - 1ull;
      const unsigned long long lo_new = (hi_new - Klo > width) ? hi_new - width : Klo;
      Khi = hi_new;
      Klo = lo_new;
    }
    const bool stop = band <= (unsigned long long)kBufCap || Klo == Khi;
    cluster.sync();  // merged arrays, parts and the leader's buffer are free again
    if (dlevel) VT_CTRACE(c, 13);
    if (stop) break;
  }
  // Gather the band into the leader; with_draw, draw over the elements above
  // it: bin below dsel, or bin dsel with a key above the band.
  {
    uint64_t* lg = cluster.map_shared_rank(c.buf, 0);
    int* lcount = cluster.map_shared_rank(&s.gcount, 0);
    const uint32_t klo_hi = (uint32_t)(Klo >> 32);
    const unsigned long long lo = Klo, hk = Khi;
    const int ds = dsel;
    float s_cur = -INFINITY, bz = 0.f;
    int bidx = INT_MAX;
    // 0: not in the set or below the band, 1: above the band, 2: in the band
    auto classify = [&](float x, float zt, int j) -> int {
      if (j >= hi || !in_pred(zt)) return 0;
      const unsigned long long K = elem_key(zt, (uint32_t)j);
      if (K < kbound) return 0;
      const int dd = slot(x, zt);
      if (dd < ds || (dd == ds && K > hk)) return 1;
      return (dd == ds && K >= lo) ? 2 : 0;
    };
    auto visit = [&](float zt, int j, int cls, uint32_t nbits) {
      if (cls == 2) {
        const int pos = atomicAdd(lcount, 1);
        if (pos < kBufCap) lg[pos] = elem_key(zt, (uint32_t)j);
      } else if (cls == 1 && with_draw && may_beat(zt, s_cur, nbits)) {
        const float sc = gumbel_score(zt, nbits);
        if (pair_better(sc, j, s_cur, bidx)) {
          s_cur = sc;
          bidx = j;
          bz = zt;
        }
      }
    };
    for_each_group<T>(
        c, [&](float gz) { return ord_key(gz) >= klo_hi; },
        [&](float* x, int, int j0) {
#pragma unroll
          for (int i = 0; i < E; i += 2) {
            const float z0 = __fmul_rn(x[i], inv_t), z1 = __fmul_rn(x[i + 1], inv_t);
            const int c0 = classify(x[i], z0, j0 + i), c1 = classify(x[i + 1], z1, j0 + i + 1);
            if ((c0 | c1) == 0) continue;
            // one SplitMix64 output serves the column pair (j0 + i, j0 + i + 1)
            const uint64_t hh = (with_draw && ((c0 | c1) & 1)) ? pair_hash(rkey, j0 + i) : 0ull;
            if (c0) visit(z0, j0 + i, c0, bits_even(hh));
            if (c1) visit(z1, j0 + i + 1, c1, bits_odd(hh));
          }
        });
    if (with_draw) {
      block_argmax(s_cur, bidx, bz, s);
      if (c.tid == 0) {
        s.part.dscore = s_cur;
        s.part.didx = bidx;
        s.part.dz = bz;
      }
    }
    VT_CTRACE(c, 14);
    cluster.sync();
    if (c.rank == 0) {
      const int n = min(s.gcount, kBufCap);
      block_sort_desc(c.buf, n);
      const int per = (n + kThreads - 1) / kThreads;
      const int i0 = min(n, c.tid * per), i1 = min(n, i0 + per);
      unsigned long long lc = 0, lm = 0;
      for (int i = i0; i < i1; ++i) {
        lc += 1;
        if (by_mass) lm += mass_fixed(key_z(c.buf[i]), m_t);
      }
      unsigned long long tot;
      const unsigned long long ex_c = block_exclusive_u64(lc, s, &tot);
      const unsigned long long ex_m = block_exclusive_u64(lm, s, &tot);
      int hit = INT_MAX;
      unsigned long long hit_c = 0, hit_m = 0;
      unsigned long long rc = acc_c + ex_c, rm = acc_m + ex_m;
      for (int i = i0; i < i1; ++i) {
        rc += 1;
        if (by_mass) rm += mass_fixed(key_z(c.buf[i]), m_t);
        if (by_mass ? (rm > target) : (rc > target)) {
          hit = i;
          hit_c = rc;
          hit_m = rm;
          break;
        }
      }
      int hmin = hit;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) hmin = min(hmin, __shfl_xor_sync(0xffffffffu, hmin, o));
      if (c.lane == 0) s.ri[c.warp] = hmin;
      __syncthreads();
      if (c.tid == 0) {
        int hh = INT_MAX;
        for (int w = 0; w < kWarps; ++w) hh = min(hh, s.ri[w]);
        s.bcast_i[0] = hh;
      }
      __syncthreads();
      const int hb = s.bcast_i[0];
      if (hb != INT_MAX && hit == hb) {
        s.sel.kb = c.buf[hb];
        s.sel.cnt_incl = hit_c;
        s.sel.mass_incl = hit_m;
        s.sel.all = 0;
      }
      if (hb == INT_MAX && c.tid == 0) {  // cannot happen: the band holds the crossing
        s.sel.kb = n > 0 ? c.buf[n - 1] : kbound;
        s.sel.cnt_incl = acc_c + n;
        s.sel.mass_incl = acc_m;
        s.sel.all = 0;
        atomicOr(&s.part.err, kErrInternal);
      }
      if (c.tid == 0) {
        s.sel.total_cnt = total_c;
        s.sel.total_mass = total_m;
        s.sel.draw_ok = 0;
      }
      if (with_draw && hb != INT_MAX) {
        // winner: the kept band prefix [0, hb] and every CTA's best above the band
        unsigned long long best = kNegInfKey;
        for (int i = c.tid; i <= hb; i += kThreads) {
          const uint64_t k = c.buf[i];
          const int j = (int)key_idx(k);
          const unsigned long long key =
              elem_key(gumbel_score(key_z(k), noise_bits(rkey, j)), (uint32_t)j);
          best = key > best ? key : best;
        }
        if (c.tid < c.C) {
          const Part* pr = cluster.map_shared_rank(&s.part, c.tid);
          if (pr->didx != INT_MAX) {
            const unsigned long long key = elem_key(pr->dscore, (uint32_t)pr->didx);
            best = key > best ? key : best;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long w = __shfl_xor_sync(0xffffffffu, best, o);
          best = w > best ? w : best;
        }
        if (c.lane == 0) s.ru[c.warp] = best;
        __syncthreads();
        if (c.tid == 0) {
          unsigned long long t = kNegInfKey;
          for (int w = 0; w < kWarps; ++w) t = s.ru[w] > t ? s.ru[w] : t;
          s.sel.win = t;
          s.sel.draw_ok = 1;
        }
      }
    }
    cluster.sync();
    out = *cluster.map_shared_rank(&s.sel, 0);
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
  for (int top = len; top > pos; top -= kThreads) {
    const int e = top - 1 - threadIdx.x;
    int2 v = make_int2(0, 0);
    const bool mine = e >= pos;
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

// Kept-set processing on the sorted candidates in the leader's buffer.
// Returns L3 (kept count); writes the drawn token and its tempered logit.
__device__ int leader_draw(Ctx& c, Smem& s, int N, int* tok, float* ztok) {
  int pass = 0;
  if (c.minp)
    for (int i = c.tid; i < N; i += kThreads) pass += minp_pass(key_z(c.buf[i]), c.m_t, c.lmp);
  const int L1 = c.minp ? block_sum_int(pass, s) : N;
  const int L2 = c.topk ? min(c.top_k, L1) : L1;
  int L3 = L2;
  if (c.topp) {
    const int per = (L2 + kThreads - 1) / kThreads;
    const int i0 = min(L2, c.tid * per), i1 = min(L2, i0 + per);
    unsigned long long lm = 0;
    for (int i = i0; i < i1; ++i) lm += mass_fixed(key_z(c.buf[i]), c.m_t);
    unsigned long long tot;
    const unsigned long long ex = block_exclusive_u64(lm, s, &tot);
    const unsigned long long Tm = (unsigned long long)((double)tot * (double)c.top_p);
    int kept = 0;
    unsigned long long run = ex;
    for (int i = i0; i < i1; ++i) {
      if (run <= Tm) ++kept;
      run += mass_fixed(key_z(c.buf[i]), c.m_t);
    }
    L3 = max(1, block_sum_int(kept, s));
  }
  float bs = -INFINITY, bz = 0.f;
  int bidx = INT_MAX;
  for (int i = c.tid; i < L3; i += kThreads) {
    const uint64_t k = c.buf[i];
    const int j = (int)key_idx(k);
    const float zt = key_z(k);
    const float sc = gumbel_score_inl(zt, noise_bits(c.rkey, j));
    if (pair_better(sc, j, bs, bidx)) {
      bs = sc;
      bidx = j;
      bz = zt;
    }
  }
  block_argmax(bs, bidx, bz, s);
  *tok = bidx;
  *ztok = bz;
  return L3;
}

// The same without top-p, on the unsorted candidates: the kept set is the
// L2 = min(top_k, min-p survivors) largest keys, found by selection.  Returns
// L2; *kk is the last kept key.
__device__ int leader_draw_unordered(Ctx& c, Smem& s, int N, int* tok, float* ztok,
                                     uint64_t* kk) {
  int pass = 0;
  if (c.minp)
    for (int i = c.tid; i < N; i += kThreads) pass += minp_pass(key_z(c.buf[i]), c.m_t, c.lmp);
  const int L1 = c.minp ? block_sum_int(pass, s) : N;
  const int L2 = max(1, c.topk ? min(c.top_k, L1) : L1);
  const uint64_t kb = block_select_desc(c.buf, N, L2, s);
  float bs = -INFINITY, bz = 0.f;
  int bidx = INT_MAX;
  for (int i = c.tid; i < N; i += kThreads) {
    const uint64_t k = c.buf[i];
    if (k < kb) continue;
    const int j = (int)key_idx(k);
    const float zt = key_z(k);
    const float sc = gumbel_score_inl(zt, noise_bits(c.rkey, j));
    if (pair_better(sc, j, bs, bidx)) {
      bs = sc;
      bidx = j;
      bz = zt;
    }
  }
  block_argmax(bs, bidx, bz, s);
  *tok = bidx;
  *ztok = bz;
  *kk = kb;
  return L2;
}

// ---------------------------------------------------------------------------
// per-row set-up shared by both kernels
// ---------------------------------------------------------------------------
// Geometry, shared-memory views and parameters of row `row` for CTA `rank` of
// a C-CTA cluster whose CTAs own `slice` elements each.
template <typename T>
__device__ RowParams init_row(Ctx& c, const SampleArgs& a, uint8_t* dsm, int row, int C,
                              int rank, int slice, uint32_t off_gmax, uint32_t off_mrg) {
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  c.C = C;
  c.rank = rank;
  c.row = row;
  c.V = a.V;
  c.slice = slice;
  c.lo = rank * slice;
  c.hi = min(c.lo + slice, a.V);
  c.ngroups = slice / Elt<T>::E;
  c.aligned = a.aligned != 0;
  c.rowp = reinterpret_cast<const T*>(a.logits) + (int64_t)row * a.ld;
  c.buf = reinterpret_cast<uint64_t*>(dsm);
  c.hcnt = reinterpret_cast<unsigned int*>(dsm);  // aliases the gather buffer
  c.gmax = reinterpret_cast<uint16_t*>(dsm + off_gmax);
  c.mmass = reinterpret_cast<unsigned long long*>(dsm + off_mrg);
  c.mcnt = reinterpret_cast<unsigned int*>(dsm + off_mrg + (kCodeSlots / C) * 8);
  const RowParams P = a.params[row];
  c.greedy = (P.flags & kRowGreedy) != 0;
  c.inv_t = P.inv_t;
  c.ax = P.inv_t * kLog2e;
  c.top_k = P.top_k;
  c.top_p = P.top_p;
  bool topp = (P.flags & kRowTopP) != 0;
  if (P.flags & kRowDecay) {  // the decayed top_p; 1 (the start) filters nothing
    c.top_p = a.decay[row].p;
    topp = c.top_p < 1.0f;
  }
  c.topk = !c.greedy && P.top_k > 1 && P.top_k < a.V;
  c.topp = !c.greedy && topp;
  c.minp = !c.greedy && (P.flags & kRowMinP) != 0;
  c.lmp = P.log_min_p;
  c.rkey = row_key(a.seeds[row], row);
  c.trace = nullptr;
  c.pen = false;
  c.bitmap = nullptr;
  c.prefix = nullptr;
  c.side_z = nullptr;
  c.stage = nullptr;
  c.xmax = 0.f;
  return P;
}

// Penalties of the slice's seen tokens: a bitmap of their positions and the
// side-list index of each bitmap word in shared memory; their penalised values
// (id order) go to shared memory after the prefixes when they fit (kSideSmem),
// else to the row's side list in global memory.  Pass A patches every group
// that holds one, and with the values in global memory each such group would
// wait on a dependent load before the stage's barrier.
template <typename T>
__device__ void setup_penalties(Ctx& c, Smem& s, const SampleArgs& a, const RowParams& P,
                                uint8_t* dsm, uint32_t off_bitmap, uint32_t off_prefix,
                                int hist_len) {
  const int2* tab = a.hist + (int64_t)c.row * a.hist_cap;
  float* zs = a.zside + (int64_t)c.row * a.hist_cap;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dsm + off_bitmap);
  uint16_t* prefix = reinterpret_cast<uint16_t*>(dsm + off_prefix);
  const int nwords = c.slice / 32;
  float* side_smem =
      reinterpret_cast<float*>(dsm + ((off_prefix + (uint32_t)nwords * 2u + 15u) & ~15u));
  for (int w = c.tid; w < nwords; w += kThreads) bitmap[w] = 0u;
  int below_lo = 0, below_hi = 0;
  for (int e = c.tid; e < hist_len; e += kThreads) {
    const int id = tab[e].x;
    below_lo += id < c.lo;
    below_hi += id < c.hi;
  }
  const int e_lo = block_sum_int(below_lo, s);
  const int e_hi = block_sum_int(below_hi, s);
  const T* row = reinterpret_cast<const T*>(c.rowp);
  float* side = e_hi - e_lo <= kSideSmem ? side_smem : zs + e_lo;
  for (int e = e_lo + c.tid; e < e_hi; e += kThreads) {
    const int2 t = tab[e];
    const int local = t.x - c.lo;
    if (local < 0 || local >= c.hi - c.lo) {  // an unsorted table never writes outside
      atomicOr(&s.part.err, kErrInternal);
      continue;
    }
    side[e - e_lo] = penalize(Elt<T>::load1(row + t.x), t.y, P);
    atomicOr(&bitmap[local >> 5], 1u << (local & 31));
  }
  __syncthreads();
  // side-list index of each word's first position: exclusive scan of popcounts
  const int per = (nwords + kThreads - 1) / kThreads;
  const int w0 = min(nwords, c.tid * per), w1 = min(nwords, w0 + per);
  unsigned long long cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bitmap[w]);
  unsigned long long tot;
  unsigned long long run = block_exclusive_u64(cnt, s, &tot);
  for (int w = w0; w < w1; ++w) {
    prefix[w] = (uint16_t)run;
    run += __popc(bitmap[w]);
  }
  c.bitmap = bitmap;
  c.prefix = prefix;
  c.side_z = side;
  c.pen = true;
  __syncthreads();
}

// ---------------------------------------------------------------------------
// kernel 1: stream every row once; finish the rows its candidates can finish
// ---------------------------------------------------------------------------
// This CTA's candidate thresholds (s.part.tau for the kept set, s.part.tau_n
// for the top-n): at least Kc (Kn) of its elements are >= them.  Up to
// kThreads, the Kc-th largest thread maximum (s.tmax); beyond, a two-round
// radix select over the bf16 lower bounds of the group maxima.  bv is the
// CTA's maximum.  All threads of the CTA call it.
__device__ __forceinline__ void cta_thresholds(const Ctx& c, Smem& s, int Kc, int Kn, float bv) {
  if (c.tid == 0) {
    s.part.tau = INFINITY;
    s.part.tau_n = INFINITY;
  }
  __syncthreads();
  if ((Kc > 0 && Kc <= kSmallK) || Kn > 0) {
    const float v = s.tmax[c.tid];
    int rank = 0;
    const float4* t4 = reinterpret_cast<const float4*>(s.tmax);
#pragma unroll 4
    for (int u = 0; u < kThreads / 4; ++u) {
      const float4 w = t4[u];
      const int b = 4 * u;
      rank += (w.x > v) || (w.x == v && b < c.tid);
      rank += (w.y > v) || (w.y == v && b + 1 < c.tid);
      rank += (w.z > v) || (w.z == v && b + 2 < c.tid);
      rank += (w.w > v) || (w.w == v && b + 3 < c.tid);
    }
    if (Kc > 0 && Kc <= kSmallK && rank == Kc - 1) s.part.tau = v;
    if (Kn > 0 && rank == Kn - 1) s.part.tau_n = v;
  }
  if (Kc > kSmallK) {
    if (Kc > c.ngroups || bv == -INFINITY) {
      if (c.tid == 0) s.part.tau = -INFINITY;
    } else {
      // The Kc-th largest group-maximum lower bound, exactly: the distance of
      // each group's order-preserving 16-bit key below the CTA maximum's, in
      // bins of 16 keys (256 bins, the last one open), then inside the chosen
      // bin by the low 4 bits.  Distances spread over many bins, so the
      // shared-memory counts rarely collide.
      auto gkey = [&](uint32_t u) -> uint32_t {
        return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
      };
      const uint32_t kmax = gkey(bf16_down(bv));
      int dsel = 0;      // chosen distance (bins of 16, then exact)
      uint32_t below = 0u;  // groups nearer the maximum than the chosen bin
      for (int round = 0; round < 2; ++round) {
        s.hist256[c.tid] = 0u;
        __syncthreads();
        for (int g = c.tid; g < c.ngroups; g += kThreads) {
          const uint32_t k = gkey(c.gmax[g]);
          const uint32_t d = k <= kmax ? kmax - k : 0u;
          if (round == 0) {
            atomicAdd(&s.hist256[d >= 255u * 16u ? 255u : d >> 4], 1u);
          } else if ((int)(d >> 4) == dsel) {
            atomicAdd(&s.hist256[d & 15u], 1u);
          }
        }
        __syncthreads();
        if (c.warp == 0) {
          // lane l holds bins 8l .. 8l+7 (ascending distance)
          uint32_t cnt[8], tot = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            cnt[q] = s.hist256[8 * c.lane + q];
            tot += cnt[q];
          }
          uint32_t inc = tot;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t w = __shfl_up_sync(0xffffffffu, inc, o);
            if (c.lane >= o) inc += w;
          }
          const uint32_t before = below + inc - tot;
          if (before < (uint32_t)Kc && below + inc >= (uint32_t)Kc) {
            uint32_t run = before;
            for (int q = 0; q < 8; ++q) {
              if (run + cnt[q] >= (uint32_t)Kc) {
                s.bcast_i[2] = 8 * c.lane + q;
                s.bcast_i[3] = (int)run;
                break;
              }
              run += cnt[q];
            }
          }
        }
        __syncthreads();
        const int bsel = s.bcast_i[2];
        below = (uint32_t)s.bcast_i[3];
        __syncthreads();  // the histogram is cleared again only after every read
        if (round == 0) {
          if (bsel == 255) {  // the open bin: every group is a candidate group
            if (c.tid == 0) s.part.tau = -INFINITY;
            break;
          }
          dsel = bsel;
        } else if (c.tid == 0) {
          const uint32_t k = kmax - (uint32_t)(dsel * 16 + bsel);
          const uint32_t u = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
          s.part.tau = bf16_val((uint16_t)u);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// pass A of a row slice: statistics while streaming it once
// ---------------------------------------------------------------------------
// A thread's group with the largest maximum, kept in registers by pass A, and
// the largest maximum of its other groups: pass B takes its candidates from
// here instead of reading the slice again whenever no other group of the
// thread can hold one (fp32 groups of 8).
struct GroupStash {
  float v[8];
  float gm = -INFINITY;      // the kept group's maximum
  float second = -INFINITY;  // the largest maximum of the thread's other groups
  int g = -1;                // the kept group (-1: none)
};

// Streams this CTA's slice (bulk copies through a ring of kStages slots in
// `ring` for aligned rows, else plain loads) and leaves in s.part its tempered
// maximum m, sum of exp(z_t - m) s, the lowest-index argmax (bv, bi) and the
// non-finite flag; s.tmax holds each thread's maximum and c.gmax each group's
// (a bf16 lower bound).  With a stash (fp32 rows), also this thread's best
// group.  Returns this CTA's maximum bv.  All threads call it.
template <typename T>
__device__ __forceinline__ float stream_stats(Ctx& c, Smem& s, uint8_t* ring,
                                              GroupStash* stash = nullptr) {
  constexpr int E = Elt<T>::E;
  // rm: this thread's running maximum (pre-temperature); rmt = fl(rm / T),
  // the tempered reference of rsum = sum of exp(z_t - rmt).
  float rm = -INFINITY, rmt = -INFINITY, rsum = 0.f, bv = -INFINITY;
  int bi = INT_MAX;
  bool nanf = false;
  auto consume = [&](float* x, int g) {
    float gm = x[0];
#pragma unroll
    for (int i = 1; i < E; ++i) gm = fmaxf(gm, x[i]);
    c.gmax[g] = bf16_down(gm);
    if constexpr (E == 8) {
      if (stash) {
        if (gm > stash->gm) {
          stash->second = fmaxf(stash->second, stash->gm);
          stash->gm = gm;
          stash->g = g;
#pragma unroll
          for (int i = 0; i < 8; ++i) stash->v[i] = x[i];
        } else {
          stash->second = fmaxf(stash->second, gm);
        }
      }
    }
    if (gm > bv) {
      int first = 0;
#pragma unroll
      for (int i = E - 1; i >= 0; --i)
        if (x[i] == gm) first = i;
      bv = gm;
      bi = c.lo + g * E + first;
    }
    if (gm > rm) {
      const float gmt = __fmul_rn(gm, c.inv_t);
      rsum = (rm == -INFINITY) ? 0.f
                               : rsum * ex2_approx(__fmul_rn(__fsub_rn(rmt, gmt), kLog2e));
      rm = gm;
      rmt = gmt;
    }
    if (rm > -INFINITY) {
      // exponentials in place, then a pairwise sum of the group.  Near zero
      // one FFMA per element, 2^(x a - rm a) with a = log2(e) / T; once the
      // reference is large, the rounding of rm a would show, and the
      // tempered difference fl(fl(x / T) - rmt) is formed instead (exact
      // where it matters, by Sterbenz).
      if (fabsf(rmt) <= 16.0f) {
        const float nb = -rm * c.ax;
#pragma unroll
        for (int i = 0; i < E; ++i) x[i] = ex2_approx(fmaf(x[i], c.ax, nb));
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i)
          x[i] = ex2_approx(__fmul_rn(__fsub_rn(__fmul_rn(x[i], c.inv_t), rmt), kLog2e));
      }
#pragma unroll
      for (int w = 1; w < E; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < E; i += 2 * w) x[i] += x[i + w];
      rsum += x[0];
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) nanf |= x[i] != x[i];
    }
  };
  if (c.aligned) {
    // bulk copies through a ring of kStages slots of kGroupsPerStage groups a
    // thread, kStages - 1 stages in flight while one is consumed
    const uint32_t bulk = ((uint32_t)(c.hi > c.lo ? c.hi - c.lo : 0) * (uint32_t)sizeof(T)) & ~15u;
    const int nstage = (c.ngroups + kThreads * kGroupsPerStage - 1) / (kThreads * kGroupsPerStage);
    const char* src = reinterpret_cast<const char*>(reinterpret_cast<const T*>(c.rowp) + c.lo);
    auto stage_bytes = [&](int k) -> uint32_t {
      const int64_t b = (int64_t)bulk - (int64_t)k * kStageBytes;
      return b <= 0 ? 0u : (b > kStageBytes ? (uint32_t)kStageBytes : (uint32_t)b);
    };
    if (c.tid == 0) {
      for (int st = 0; st < kStages; ++st) mbar_init(&s.full[st], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (c.tid == 0) {
      for (int k = 0; k < min(kStages, nstage); ++k) {
        const uint32_t by = stage_bytes(k);
        if (by) {
          mbar_arrive_expect_tx(&s.full[k], by);
          bulk_copy_g2s(ring + k * kStageBytes, src + (size_t)k * kStageBytes, by, &s.full[k]);
        }
      }
    }
    for (int k = 0; k < nstage; ++k) {
      const int slot = k % kStages;
      const uint32_t by = stage_bytes(k);
      if (by && !mbar_wait_bounded(&s.full[slot], (uint32_t)((k / kStages) & 1)))
        atomicOr(&s.part.err, kErrTimeout);
#pragma unroll
      for (int gi = 0; gi < kGroupsPerStage; ++gi) {
      const int gs = gi * kThreads + c.tid;  // the group's place in the stage
      const int g = k * kThreads * kGroupsPerStage + gs;
      if (g < c.ngroups) {
        float x[E];
        if ((uint32_t)(gs + 1) * kGroupBytes <= by) {
          const uint4* q = reinterpret_cast<const uint4*>(ring + slot * kStageBytes) + 2 * gs;
          if constexpr (E == 8) {
            const uint4 u0 = q[0], u1 = q[1];
            x[0] = __uint_as_float(u0.x); x[1] = __uint_as_float(u0.y);
            x[2] = __uint_as_float(u0.z); x[3] = __uint_as_float(u0.w);
            x[4] = __uint_as_float(u1.x); x[5] = __uint_as_float(u1.y);
            x[6] = __uint_as_float(u1.z); x[7] = __uint_as_float(u1.w);
          } else {
            const uint4 u0 = q[0], u1 = q[1];
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              x[2 * i] = __uint_as_float(w[i] << 16);
              x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
          }
          patch_group<T>(c, g, x);
        } else {
          load_group<T>(c, g, x);  // the ragged tail, from global memory
        }
        consume(x, g);
      }
      }
      __syncthreads();  // slot free
      if (s.part.err & kErrTimeout) {
        // a wait ran out: issue nothing more, and wait once more (bounded) for
        // the copies still in flight (stages k .. k + kStages - 1) before the
        // ring is left; the row's results are void and the error word says so
        if (c.tid == 0) {
          for (int q = k; q < min(nstage, k + kStages); ++q)
            if (stage_bytes(q)) (void)mbar_wait_bounded(&s.full[q % kStages], (uint32_t)((q / kStages) & 1));
        }
        __syncthreads();
        break;
      }
      if (c.tid == 0 && k + kStages < nstage) {
        const uint32_t nb = stage_bytes(k + kStages);
        if (nb) {
          mbar_arrive_expect_tx(&s.full[slot], nb);
          bulk_copy_g2s(ring + slot * kStageBytes, src + (size_t)(k + kStages) * kStageBytes,
                        nb, &s.full[slot]);
        }
      }
    }
  } else {
    for (int g = c.tid; g < c.ngroups; g += kThreads) {
      float x[E];
      load_group<T>(c, g, x);
      consume(x, g);
    }
  }
  const bool nonfin = nanf || (rsum != rsum) || rm == INFINITY;
  s.tmax[c.tid] = rm;
  float m = rmt, sm = rsum;  // partials combine in tempered units
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
    lse_combine(m, sm, m2, s2, kLog2e);
  }
  float dz = 0.f;
  block_argmax(bv, bi, dz, s);  // also a barrier: s.tmax is complete after it
  const int nf = __syncthreads_or(nonfin);
  // (rows handed over after their statistics take no thresholds here)
  if (c.lane == 0) {
    s.rf[c.warp] = m;
    s.rf[kWarps + c.warp] = sm;
  }
  __syncthreads();
  if (c.tid == 0) {
    float mm = -INFINITY, ss = 0.f;
    for (int w = 0; w < kWarps; ++w) lse_combine(mm, ss, s.rf[w], s.rf[kWarps + w], kLog2e);
    s.part.m = mm;
    s.part.s = ss;
    s.part.bv = bv;
    s.part.bi = bi;
    s.part.nonfinite = nf;
  }
  __syncthreads();
  return bv;
}

// Top-p decay after the row's sampled token [TensorRT-LLM "Sampling", top-p
// decay]: back to the initial top_p when the token is the reset id, else
// max(top_p * decay, top_p_min), in fp32.  One thread of the row calls it.
__device__ __forceinline__ void decay_top_p(const SampleArgs& a, int row, int tok) {
  const RowParams& P = a.params[row];
  if (!(P.flags & kRowDecay)) return;
  DecayState& d = a.decay[row];
  const float q = __fmul_rn(d.p, d.decay);
  d.p = tok == d.reset_id ? P.top_p : (q < d.p_min ? d.p_min : q);
}

// Outputs of a row whose statistics make it unsampleable (non-finite values,
// or no finite value): token -1, NaN log-probs, the status; the seed still
// advances and the top-p decay state stays.  The row's leader CTA calls it.
__device__ __forceinline__ void write_bad_row(const SampleArgs& a, const Smem& s, int row,
                                              int status) {
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
    if (s.rs.err) atomicOr(a.err_word, s.rs.err);
  }
}

// The row's statistics from every CTA's pass-A partials (warp 0; the caller
// synchronises): tempered maximum, sum and its log, argmax, flags, and the
// smallest candidate thresholds.
__device__ __forceinline__ void cluster_stats(const Ctx& c, Smem& s, cg::cluster_group& cluster) {
  if (c.warp == 0) {
    float m = -INFINITY, sm = 0.f, bv = -INFINITY, tau = INFINITY, tau_n = INFINITY;
    int bi = INT_MAX, nf = 0, er = 0;
    if (c.lane < c.C) {
      const Part* p = cluster.map_shared_rank(&s.part, c.lane);
      m = p->m;
      sm = p->s;
      bv = p->bv;
      bi = p->bi;
      nf = p->nonfinite;
      er = p->err;
      tau = p->tau;
      tau_n = p->tau_n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
      lse_combine(m, sm, m2, s2, kLog2e);
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (pair_better(v2, i2, bv, bi)) {
        bv = v2;
        bi = i2;
      }
      nf |= __shfl_xor_sync(0xffffffffu, nf, o);
      er |= __shfl_xor_sync(0xffffffffu, er, o);
      tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, o));
      tau_n = fminf(tau_n, __shfl_xor_sync(0xffffffffu, tau_n, o));
    }
    if (c.lane == 0) {
      // m is the tempered row maximum fl(max / T) (rounding is monotone)
      s.rs.m_t = m;
      s.rs.S = sm;
      s.rs.lnS = logf(sm);
      s.rs.bv = bv;
      s.rs.bi = bi;
      s.rs.nonfinite = nf || m == INFINITY;
      s.rs.err = er;
      s.rs.tau = tau;
      s.rs.tau_n = tau_n;
    }
  }
}

template <typename T>
// fp32 rows (penalties and 4-byte logits) run at 2 CTAs an SM with the
// registers that frees; bf16 rows at 4, which keeps every row of a large batch
// resident beside the selection kernel's CTAs
__global__ void __launch_bounds__(kThreads, (sizeof(T) == 4 ? 2 : 4))
    sample_kernel(const SampleArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ Smem s;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int E = Elt<T>::E;

  Ctx c;
  const int C = (int)cluster_nctarank();
  const int row = a.rows ? a.rows[blockIdx.x / C] : (int)(blockIdx.x / C);
  const RowParams P = init_row<T>(c, a, dsm, row, C, (int)cluster_ctarank(), a.slice,
                                  a.off_gmax, a.off_mrg);
  c.trace = a.trace ? a.trace + ((size_t)row * C + c.rank) * kTraceSlots : nullptr;
  const int n = a.n_logprobs;
  const int hist_len = a.hist_len[c.row];
  VT_TRACE(0);

  if (c.tid == 0) {
    s.part.err = 0;
    s.nloc = 0;
    s.gcount = 0;
  }

  if (a.pen_smem && (P.flags & kRowPenalty) != 0 && hist_len > 0)
    setup_penalties<T>(c, s, a, P, dsm, a.off_bitmap, a.off_prefix, hist_len);

  // ---- pass A: stream the slice ----------------------------------------------
  // Candidates the kept set may need (K_main) and the top-n alone (n).
  int K_main = c.greedy ? n : max(n, c.topk ? c.top_k : ((c.topp || c.minp) ? kDefaultCand : 0));
  bool topk_beyond = false;
  if (K_main > kBufCap) {
    K_main = n;
    topk_beyond = true;
  }
  GroupStash stash;
  const float cta_max = stream_stats<T>(c, s, reinterpret_cast<uint8_t*>(c.buf),
                                        sizeof(T) == 4 ? &stash : nullptr);
  {
    // (rows handed over after their statistics take no thresholds)
    const int Kc = a.early ? 0 : (K_main + c.C - 1) / c.C;
    const int Kn = a.early ? 0 : (n + c.C - 1) / c.C;
    cta_thresholds(c, s, Kc, Kn, cta_max);
  }
  VT_TRACE(2);
  cluster.sync();  // (1) pass-A partials and thresholds visible
  VT_TRACE(3);
  cluster_stats(c, s, cluster);
  __syncthreads();
  c.m_t = s.rs.m_t;
  c.lnS = s.rs.lnS;
  const int status0 = s.rs.nonfinite ? kRowNonfinite : (s.rs.m_t == -INFINITY ? kRowEmpty : kRowOk);
  const bool leader = c.rank == 0;
  int32_t* out_ids = n > 0 ? a.out_topk_ids + (int64_t)c.row * n : nullptr;
  float* out_lps = n > 0 ? a.out_topk_logprobs + (int64_t)c.row * n : nullptr;

  if (status0 != kRowOk) {
    cluster.sync();  // nobody reads another CTA's shared memory after this
    if (leader) write_bad_row(a, s, c.row, status0);
    return;
  }

  // ---- rows routed to the selection kernel: hand over after the statistics ----
  if (a.early) {
    cluster.sync();  // every CTA has read the others' pass-A partials
    if (leader && c.tid == 0) {
      SlowRow r;
      r.m_t = c.m_t;
      r.lnS = c.lnS;
      r.xmax = s.rs.bv;
      r.bi_topn = (uint32_t)s.rs.bi | (n == 0 ? 0x80000000u : 0u);
      a.slow[c.row] = r;
      a.slow_list[atomicAdd(a.slow_ctl, 1u)] = c.row;
      if (s.rs.err) atomicOr(a.err_word, s.rs.err);
    }
    VT_TRACE(15);
    return;
  }
  // ---- pass B: candidates at or above the cluster threshold ----------------
  // A top-p row without top-k keeps at least p * S elements (none weighs more
  // than the maximum): past the buffer it cannot stay on the candidates, so
  // only the top-n ones are collected.
  bool likely_slow = topk_beyond;
  if (!c.greedy && !c.topk && c.topp && (double)c.top_p * (double)s.rs.S > (double)kBufCap)
    likely_slow = true;
  if (!c.greedy && !c.topk && !c.topp && !c.minp) likely_slow = true;  // unfiltered draw
  const int K_need = likely_slow ? n : K_main;
  const float tau = likely_slow ? s.rs.tau_n : s.rs.tau;
  const bool complete = K_need > 0 && tau == -INFINITY;
  {
    int my_n = 0, my_minp = 0;
    unsigned long long my_mass = 0;
    if (K_need > 0) {
      const float tau_t = __fmul_rn(tau, c.inv_t);
      auto collect = [&](float* x, int, int j0) {
            uint32_t take = 0u;
#pragma unroll
            for (int i = 0; i < E; ++i) {
              const float zt = __fmul_rn(x[i], c.inv_t);
              x[i] = zt;
              if (j0 + i < c.hi && zt >= tau_t && zt > -INFINITY) take |= 1u << i;
            }
            if (take == 0u) return;
            int pos = atomicAdd(&s.nloc, __popc(take));  // one atomic per group
#pragma unroll
            for (int i = 0; i < E; ++i) {
              if (take & (1u << i)) {
                if (pos < kBufCap) c.buf[pos] = elem_key(x[i], (uint32_t)(j0 + i));
                ++pos;
                ++my_n;
                my_mass += mass_fixed(x[i], c.m_t);
                if (c.minp && minp_pass(x[i], c.m_t, c.lmp)) ++my_minp;
              }
            }
          };
      // fp32: the stashed group serves unless another group of this thread
      // reaches the threshold (fl(max / T) bounds every tempered value of it)
      bool from_stash = false;
      if constexpr (E == 8) {
        from_stash = !(__fmul_rn(stash.second, c.inv_t) >= tau_t);
        if (from_stash && stash.g >= 0 && __fmul_rn(stash.gm, c.inv_t) >= tau_t)
          collect(stash.v, stash.g, c.lo + stash.g * E);
      }
      if (!from_stash) for_each_group<T>(c, [&](float gz) { return gz >= tau_t; }, collect);
    }
    // one combined CTA reduction of (count, min-p count, mass)
    my_n = warp_sum_i(my_n);
    my_minp = warp_sum_i(my_minp);
    my_mass = warp_sum_u64(my_mass);
    if (c.lane == 0) {
      s.ri[c.warp] = my_n;
      s.ri[kWarps + c.warp] = my_minp;
      s.ru[c.warp] = my_mass;
    }
    __syncthreads();
    if (c.tid == 0) {
      int tn = 0, tm = 0;
      unsigned long long tmass = 0;
      for (int w = 0; w < kWarps; ++w) {
        tn += s.ri[w];
        tm += s.ri[kWarps + w];
        tmass += s.ru[w];
      }
      s.part.ncand = tn;
      s.part.ncand_minp = tm;
      s.part.cand_mass = tmass;
    }
  }
  VT_TRACE(6);
  cluster.sync();  // (2) candidate counts visible
  VT_TRACE(7);
  if (c.warp == 0) {
    int nc = 0, nm = 0, ov = 0;
    unsigned long long mass = 0;
    if (c.lane < c.C) {
      const Part* p = cluster.map_shared_rank(&s.part, c.lane);
      nc = p->ncand;
      nm = p->ncand_minp;
      mass = p->cand_mass;
      ov = nc > kBufCap;
    }
    int inc = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, inc, o);
      if (c.lane >= o) inc += w;
    }
    const int off = __shfl_sync(0xffffffffu, inc - nc, c.rank);
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    nm = warp_sum_i(nm);
    mass = warp_sum_u64(mass);
    ov = warp_sum_i(ov);
    if (c.lane == 0) {
      s.rs.nc = tot;
      s.rs.nc_minp = nm;
      s.rs.cand_mass = mass;
      s.rs.push_off = off;
      s.rs.overflow = ov;
    }
  }
  __syncthreads();
  const int nc = s.rs.nc;
  const bool cand_ok = K_need > 0 ? (nc <= kBufCap && !s.rs.overflow) : true;
  const bool topn_ok = n == 0 || (cand_ok && nc >= n);
  // The kept prefix is known from the candidates when every min-p survivor is
  // a candidate, or when top-k ends inside them.  A top-p row needs the exact
  // mass of the survivors it renormalises over, so it stays on the candidates
  // only when they hold every survivor of min-p and top-k.
  const bool surv_inside = complete || (c.minp && s.rs.nc_minp < nc);
  const bool L2_inside = surv_inside || (c.topk && !topk_beyond && c.top_k <= nc);
  bool fast;
  if (c.greedy) {
    fast = topn_ok;
  } else {
    if (!c.topk && !c.topp && !c.minp)
      fast = complete && cand_ok;
    else
      fast = cand_ok && L2_inside;
    fast = fast && topn_ok && K_need > 0;
  }
  // every CTA pushes its candidates into the leader's buffer when they fit
  if (cand_ok && nc > 0 && (fast || topn_ok) && c.rank > 0) {
    uint64_t* lb = cluster.map_shared_rank(c.buf, 0);
    const int mine = min(s.nloc, kBufCap);
    const int off = s.rs.push_off;
    for (int i = c.tid; i < mine; i += kThreads) lb[off + i] = c.buf[i];
  }
  cluster.sync();  // (3) gathered; partials read
  VT_TRACE(8);

  if (fast) {
    if (!leader) {
      VT_TRACE(15);
      return;
    }
    const int N = nc;
    int tok;
    float ztok;
    int L3;
    uint64_t kk = 0ull;  // the last kept key
    if (c.topp) {
      // top-p needs the masses in order: the whole candidate set sorted
      block_sort_desc(c.buf, N);
      for (int t = c.tid; t < n; t += kThreads) {
        const uint64_t k = c.buf[t];
        out_ids[t] = (int)key_idx(k);
        out_lps[t] = (key_z(k) - c.m_t) - c.lnS;
      }
      L3 = leader_draw(c, s, N, &tok, &ztok);
      kk = c.buf[L3 - 1];
    } else {
      // no order beyond the top-n: the kept boundary is a selection
      if (n > 0) {
        uint64_t* top = reinterpret_cast<uint64_t*>(s.tmax);
        block_top_desc(c.buf, N, n, top, s);
        for (int t = c.tid; t < n; t += kThreads) {
          const uint64_t k = top[t];
          out_ids[t] = (int)key_idx(k);
          out_lps[t] = (key_z(k) - c.m_t) - c.lnS;
        }
      }
      if (c.greedy) {
        tok = s.rs.bi;
        ztok = c.m_t;
        L3 = 1;
      } else {
        L3 = leader_draw_unordered(c, s, N, &tok, &ztok, &kk);
      }
    }
    if (c.tid == 0) {
      a.out_tokens[c.row] = tok;
      if (a.out_logprobs) a.out_logprobs[c.row] = (ztok - c.m_t) - c.lnS;
      a.row_status[c.row] = kRowOk;
      a.dbg_kth_value[c.row] = c.greedy ? c.m_t : key_z(kk);
      a.dbg_kth_index[c.row] = c.greedy ? tok : (int)key_idx(kk);
      a.dbg_kept[c.row] = L3;
      a.seeds[c.row] += kSeedStep;
      decay_top_p(a, c.row, tok);
      if (s.rs.err) atomicOr(a.err_word, s.rs.err);
    }
    VT_TRACE(9);
    if (a.update_counts) {
      __syncthreads();
      append_token(a.hist + (int64_t)c.row * a.hist_cap, a.hist_len + c.row, a.hist_cap, tok, s,
                   a.row_status + c.row);
    }
    VT_TRACE(15);
    return;
  }
  // ---- rows the candidates cannot finish go to the selection kernel ---------
  if (leader) {
    if (n > 0 && topn_ok) {
      uint64_t* top = reinterpret_cast<uint64_t*>(s.tmax);
      block_top_desc(c.buf, nc, n, top, s);
      for (int t = c.tid; t < n; t += kThreads) {
        const uint64_t k = top[t];
        out_ids[t] = (int)key_idx(k);
        out_lps[t] = (key_z(k) - c.m_t) - c.lnS;
      }
    }
    if (c.tid == 0) {
      SlowRow r;
      r.m_t = c.m_t;
      r.lnS = c.lnS;
      r.xmax = s.rs.bv;
      r.bi_topn = (uint32_t)s.rs.bi | ((n == 0 || topn_ok) ? 0x80000000u : 0u);
      a.slow[c.row] = r;
      a.slow_list[atomicAdd(a.slow_ctl, 1u)] = c.row;
      if (s.rs.err) atomicOr(a.err_word, s.rs.err);
    }
  }
  VT_TRACE(15);
}

// ---------------------------------------------------------------------------
// selection on bf16 codes (selection kernel, bf16 rows without penalties)
// ---------------------------------------------------------------------------
// Every element of one bf16 code has the same tempered value and mass, so the
// survivors counted per code slot (slot = code(max) - code(x)) settle the kept
// set exactly: the kept count of the boundary slot follows from its count and
// its one per-element mass, and inside a slot the order is by index.  The
// draw's best element of a slot is the one with the largest noise bits
// (lowest index on ties), so the main pass keeps, per slot, only a count and
// the largest noise bits.  The leader then walks the 4096 slots (top-n, top-k,
// top-p over the top-k survivors, min-p per slot) and finds the best wholly
// kept slot; one index-ordered pass settles the kept prefix of the boundary
// slot, the index of the winning element and the top-n.  The tiny slot
// (|x| < 2^-12 and both zeros) and the catch-all hold several values: their
// elements are counted, summed and drawn one by one (shared atomics; they are
// rare).  A boundary inside one of them, a top-n that reaches -inf, or two
// slots with the same best score leave the row to the generic selection
// (returns false before any output; every CTA of the cluster returns the same).

// One element of the tiny (w = 0) or catch-all (w = 1) slot.
__device__ __noinline__ void code_special(Part& pt, int w, uint32_t u, int j, uint32_t bits,
                                          float inv_t, float m_t, bool minp, double lmp,
                                          bool draw) {
  const float zt = __fmul_rn(__uint_as_float(u << 16), inv_t);
  atomicAdd(&pt.sp_all[w], 1ull);
  if (minp && !minp_pass(zt, m_t, lmp)) return;
  atomicAdd(&pt.sp_cnt[w], 1ull);
  atomicAdd(&pt.sp_mass[w], mass_fixed(zt, m_t));
  if (draw) atomicMax(&pt.sp_key[w], elem_key(gumbel_score(zt, bits), (uint32_t)j));
}

// A fast approximation of the Gumbel score (for choosing where to compute
// the exact one): z - ln(-ln u), u = (b + 1/2) 2^-24.
__device__ __forceinline__ float approx_score(float z, uint32_t b) {
  const float u = (float)(2u * b + 1u) * 0x1p-25f;
  return z - __logf(-__logf(u));
}

template <typename T>
__device__ __forceinline__ bool code_row(Ctx& c, Smem& s, const SampleArgs& a,
                                      cg::cluster_group& cluster, bool topn_done,
                                      uint8_t* code_mem) {
  if constexpr (sizeof(T) != 2) {
    return false;
  } else {
    const int n = a.n_logprobs;
    const bool want_topn = n > 0 && !topn_done;
    const bool draw = !c.greedy;
    const bool leader = c.rank == 0;
    const int tid = c.tid, lane = c.lane, warp = c.warp, C = c.C, rank = c.rank;
    unsigned int* hc = reinterpret_cast<unsigned int*>(code_mem);  // counts per slot
    unsigned int* hb = hc + kCodeSlots;                            // best noise bits + 1
    unsigned int* mc = c.mcnt;                                     // merged, this CTA's range
    unsigned int* mb = reinterpret_cast<unsigned int*>(c.mmass);
    const int nb = kCodeSlots / C, b0 = rank * nb;
    const int cmax = code16(__float_as_uint(c.xmax) >> 16);
    const int tiny = (cmax >= 0 && cmax < kCodeSlots - 1) ? cmax : -1;
    constexpr int kCatch = kCodeSlots - 1;
    const float m_t = c.m_t, inv_t = c.inv_t, lnS = c.lnS, top_p = c.top_p;
    const bool minp = c.minp, topk = c.topk, topp = c.topp;
    const int top_k = c.top_k;
    const double lmp = c.lmp;
    const int hi = c.hi, lo = c.lo, ngroups = c.ngroups, row = c.row;
    const uint64_t rkey = c.rkey;
    // the 8 words (16 bf16) of group g: from the staged slice, else from global
    // memory (a group reaching past the row end reads -inf there)
    const uint4* stage = c.stage;
    const uint16_t* gsrc = reinterpret_cast<const uint16_t*>(c.rowp) + lo;
    auto group_words = [&](int g, uint32_t* w) {
      uint4 v0, v1;
      if (stage) {
        v0 = stage[2 * g];
        v1 = stage[2 * g + 1];
      } else if (lo + (g + 1) * 16 <= hi) {
        const uint4* q = reinterpret_cast<const uint4*>(gsrc + g * 16);
        v0 = __ldg(q);
        v1 = __ldg(q + 1);
      } else {
        uint32_t h[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) h[e] = lo + g * 16 + e < hi ? (uint32_t)__ldg(gsrc + g * 16 + e) : 0xFF80u;
        v0 = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
        v1 = make_uint4(h[8] | h[9] << 16, h[10] | h[11] << 16, h[12] | h[13] << 16,
                        h[14] | h[15] << 16);
      }
      w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
      w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
    };

    for (int b = tid; b < 2 * kCodeSlots; b += kThreads) hc[b] = 0u;
    if (tid < 2) {
      s.part.sp_all[tid] = 0ull;
      s.part.sp_cnt[tid] = 0ull;
      s.part.sp_mass[tid] = 0ull;
      s.part.sp_key[tid] = 0ull;
    }
    if (leader && tid == 0) {
      s.gcount = 0;
      s.gcount2 = 0;
    }
    __syncthreads();
    VT_CTRACE(c, 4);

    // ---- pass 1: counts and best noise bits per slot --------------------------
    const int ngroups_live = min(ngroups, (hi - lo + 15) / 16);  // groups holding row elements
    for (int g = tid; g < ngroups_live; g += kThreads) {
      uint32_t w[8];
      group_words(g, w);
      const int j0 = lo + g * 16;
      // slots of the 16 elements first (no branches), then the updates
      int sl[16];
      unsigned int special = 0u;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t u = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
        const int d = cmax - code16(u);
        const int v = d < kCatch ? d : kCatch;
        const bool live = u != 0xFF80u && j0 + e < hi;  // -inf is never a survivor
        sl[e] = live ? v : -1;
        special |= (live && (v == tiny || v == kCatch)) ? (1u << e) : 0u;
      }
      uint32_t bits[16];
      if (draw) {
        // SplitMix64 counter of the column pair (j0 + 2q, j0 + 2q + 1)
        const uint64_t base = rkey + kSeedStep * ((uint64_t)(j0 >> 1) + 1ull);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint64_t h = sm64_mix(base + kSeedStep * (uint64_t)q);
          bits[2 * q] = bits_even(h);
          bits[2 * q + 1] = bits_odd(h);
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (sl[e] < 0 || (special >> e) & 1u) continue;
        atomicAdd(&hc[sl[e]], 1u);
        if (draw) atomicMax(&hb[sl[e]], bits[e] + 1u);
      }
      // (element indices fixed at compile time: the arrays stay in registers)
      if (special) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          if ((special >> e) & 1u) {
            const uint32_t u = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
            code_special(s.part, sl[e] == tiny ? 0 : 1, u, j0 + e, draw ? bits[e] : 0u, inv_t,
                         m_t, minp, lmp, draw);
          }
        }
      }
    }
    VT_CTRACE(c, 12);
    cluster.sync();  // (a) slot counts and special parts complete

    // ---- special totals, then merge this CTA's slot range --------------------
    unsigned long long sp_all0, sp_all1, sp_cnt0, sp_cnt1, sp_m0, sp_m1, sp_k0, sp_k1;
    {
      unsigned long long v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (lane < C) {
        const Part* pr = cluster.map_shared_rank(&s.part, lane);
        v[0] = pr->sp_all[0];
        v[1] = pr->sp_all[1];
        v[2] = pr->sp_cnt[0];
        v[3] = pr->sp_cnt[1];
        v[4] = pr->sp_mass[0];
        v[5] = pr->sp_mass[1];
        v[6] = pr->sp_key[0];
        v[7] = pr->sp_key[1];
      }
#pragma unroll
      for (int q = 0; q < 6; ++q) v[q] = warp_sum_u64(v[q]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x6 = __shfl_xor_sync(0xffffffffu, v[6], o);
        const unsigned long long x7 = __shfl_xor_sync(0xffffffffu, v[7], o);
        v[6] = x6 > v[6] ? x6 : v[6];
        v[7] = x7 > v[7] ? x7 : v[7];
      }
      sp_all0 = v[0];
      sp_all1 = v[1];
      sp_cnt0 = v[2];
      sp_cnt1 = v[3];
      sp_m0 = v[4];
      sp_m1 = v[5];
      sp_k0 = v[6];
      sp_k1 = v[7];
    }
    // (nb is a multiple of kThreads: 8 slots of a thread per round, every
    // CTA's values for them loaded before any is combined)
    for (int b = tid; b < nb; b += 8 * kThreads) {
      unsigned int sc[8], sbm[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        sc[u] = 0u;
        sbm[u] = 0u;
      }
      for (int r = 0; r < C; ++r) {
        const unsigned int* hr = cluster.map_shared_rank(hc, r) + b0;
        unsigned int cnt[8], bst[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int bb = b + u * kThreads;
          cnt[u] = bb < nb ? hr[bb] : 0u;
          bst[u] = bb < nb ? hr[kCodeSlots + bb] : 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sc[u] += cnt[u];
          sbm[u] = bst[u] > sbm[u] ? bst[u] : sbm[u];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int bb = b + u * kThreads;
        if (bb < nb) {
          mc[bb] = sc[u];
          mb[bb] = sbm[u];
        }
      }
    }
    __syncthreads();
    VT_CTRACE(c, 11);

    // ---- the walk, distributed: each CTA walks its own slot range ------------
    // slot sl: count of finite elements, of survivors, and the survivors' mass
    auto zq = [&](int sl) { return __fmul_rn(code_value(cmax - sl), inv_t); };
    auto vals = [&](int sl, unsigned int& na, unsigned int& ns, unsigned long long& ms) {
      if (sl == tiny) {
        na = (unsigned int)sp_all0;
        ns = (unsigned int)sp_cnt0;
        ms = sp_m0;
        return;
      }
      if (sl == kCatch) {
        na = (unsigned int)sp_all1;
        ns = (unsigned int)sp_cnt1;
        ms = sp_m1;
        return;
      }
      na = mc[sl - b0];
      ns = 0u;
      ms = 0ull;
      if (na != 0u) {
        const float z = zq(sl);
        if (!minp || minp_pass(z, m_t, lmp)) {
          ns = na;
          ms = (unsigned long long)na * mass_fixed(z, m_t);
        }
      }
    };
    // mass of the first k survivors of slot sl (regular: k equal masses)
    auto part_mass = [&](int sl, unsigned int k, unsigned int ns, unsigned long long ms) {
      if (k == ns) return ms;
      return (unsigned long long)k * mass_fixed(zq(sl), m_t);
    };
    const int per_t = (nb + kThreads - 1) / kThreads;  // contiguous slots per thread
    const int t0 = min(b0 + nb, b0 + tid * per_t), t1 = min(b0 + nb, t0 + per_t);
    unsigned long long t_all = 0, t_cnt = 0, t_mass = 0;
    int t_last = -1;
    for (int sl = t0; sl < t1; ++sl) {
      unsigned int na, ns;
      unsigned long long ms;
      vals(sl, na, ns, ms);
      t_all += na;
      t_cnt += ns;
      t_mass += ms;
      if (ns != 0u) t_last = sl;
    }
    unsigned long long r_all, r_cnt, r_mass;
    const unsigned long long x_all = block_exclusive_u64(t_all, s, &r_all);
    const unsigned long long x_cnt = block_exclusive_u64(t_cnt, s, &r_cnt);
    const unsigned long long x_mass = block_exclusive_u64(t_mass, s, &r_mass);
    int lastw = t_last;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastw = max(lastw, __shfl_xor_sync(0xffffffffu, lastw, o));
    if (lane == 0) s.ri[warp] = lastw;
    __syncthreads();
    if (tid == 0) {
      int lm = -1;
      for (int w = 0; w < kWarps; ++w) lm = max(lm, s.ri[w]);
      s.part.rng_all = r_all;
      s.part.rng_cnt = r_cnt;
      s.part.rng_mass = r_mass;
      s.part.rng_last = lm;
      if (leader) {  // the leader's walk record starts clean
        s.cw.fallback = 0;
        s.cw.slot = -1;
        s.cw.kp = 0;
        s.cw.above = 0ull;
        s.cw.slot_n = -1;
        s.cw.kn = 0;
        s.cw.k_slot = -1;
        s.cw.k_kept = 0;
        s.cw.k_mass = 0ull;
      }
    }
    cluster.sync();  // (w1) range totals visible
    // prefix of the ranges before mine, and the row totals
    unsigned long long p_all = 0, p_cnt = 0, p_mass = 0, tot_all = 0, tot_cnt = 0, tot_mass = 0;
    int last_slot = -1;
    for (int r = 0; r < C; ++r) {
      const Part* pr = cluster.map_shared_rank(&s.part, r);
      if (r < rank) {
        p_all += pr->rng_all;
        p_cnt += pr->rng_cnt;
        p_mass += pr->rng_mass;
      }
      tot_all += pr->rng_all;
      tot_cnt += pr->rng_cnt;
      tot_mass += pr->rng_mass;
      last_slot = max(last_slot, pr->rng_last);
    }
    CodeWalk* lw = cluster.map_shared_rank(&s.cw, 0);
    const unsigned long long e_all = p_all + x_all, e_cnt = p_cnt + x_cnt, e_mass = p_mass + x_mass;
    // top-n over every finite element
    if (want_topn) {
      const unsigned long long tg = (unsigned long long)(n - 1);
      unsigned long long run = e_all;
      for (int sl = t0; sl < t1; ++sl) {
        unsigned int na, ns;
        unsigned long long ms;
        vals(sl, na, ns, ms);
        if (run <= tg && run + na > tg) {
          lw->slot_n = sl;
          lw->kn = (int)(tg + 1 - run);
          // every element up to and including this slot is gathered
          if (sl == tiny || sl == kCatch || run + na > (unsigned long long)kBufCap) lw->fallback = 1;
        }
        run += na;
      }
    }
    // top-k by count over the survivors; without top-p it is the boundary
    const bool k_active = draw && topk && tot_cnt > (unsigned long long)(top_k - 1);
    if (k_active) {
      const unsigned long long tg = (unsigned long long)(top_k - 1);
      unsigned long long run = e_cnt, runm = e_mass;
      for (int sl = t0; sl < t1; ++sl) {
        unsigned int na, ns;
        unsigned long long ms;
        vals(sl, na, ns, ms);
        if (run <= tg && run + ns > tg) {
          const unsigned int kk = (unsigned int)(tg + 1 - run);
          if (sl == tiny || sl == kCatch || na > (unsigned int)kBufCap) {
            lw->fallback = 1;  // a boundary slot is gathered whole
          } else {
            lw->k_slot = sl;
            lw->k_kept = (int)kk;
            lw->k_mass = runm + part_mass(sl, kk, ns, ms);
            if (!topp) {
              lw->slot = sl;
              lw->kp = (int)kk;
              lw->above = run;
            }
          }
        }
        run += ns;
        runm += ms;
      }
    }
    if (draw && topp) {
      int slot_k = -1;
      unsigned int kk = 0u;
      unsigned long long W = tot_mass, e_tm = e_mass;
      if (k_active) {
        cluster.sync();  // (w1b) the top-k boundary is known
        slot_k = lw->k_slot;
        kk = (unsigned int)lw->k_kept;
        W = lw->k_mass;
        // survivors' masses truncated to the top-k set
        unsigned long long tm = 0ull;
        for (int sl = t0; sl < t1 && sl <= slot_k; ++sl) {
          unsigned int na, ns;
          unsigned long long ms;
          vals(sl, na, ns, ms);
          tm += sl < slot_k ? ms : part_mass(sl, kk, ns, ms);
        }
        unsigned long long r_tm;
        const unsigned long long x_tm = block_exclusive_u64(tm, s, &r_tm);
        if (tid == 0) s.part.rng_tmass = r_tm;
        cluster.sync();  // (w1c) truncated range totals visible
        unsigned long long p_tm = 0ull;
        for (int r = 0; r < rank; ++r) p_tm += cluster.map_shared_rank(&s.part, r)->rng_tmass;
        e_tm = p_tm + x_tm;
      }
      const unsigned long long tgt_m = (unsigned long long)((double)W * (double)top_p);
      // the boundary element is the first whose inclusive mass exceeds the
      // target; its slot is the first whose inclusive mass does
      unsigned long long A = e_tm, run = e_cnt;
      for (int sl = t0; sl < t1; ++sl) {
        if (slot_k >= 0 && sl > slot_k) break;
        unsigned int na, ns;
        unsigned long long ms;
        vals(sl, na, ns, ms);
        const unsigned int nc = (slot_k >= 0 && sl == slot_k) ? kk : ns;
        if (nc == 0u) continue;
        const unsigned long long mc2 = part_mass(sl, nc, ns, ms);
        if (A <= tgt_m && A + mc2 > tgt_m) {
          if (sl == tiny || sl == kCatch || na > (unsigned int)kBufCap) {
            lw->fallback = 1;  // a boundary slot is gathered whole
          } else {
            // kq = floor((tgt_m - A) / mass) + 1, below the slot's count: a
            // float quotient corrected to the exact one by integer products
            const unsigned long long num = tgt_m - A, den = mass_fixed(zq(sl), m_t);
            unsigned long long q = (unsigned long long)__fdiv_rz((float)num, (float)den);
            while (q > 0ull && q * den > num) --q;
            while ((q + 1ull) * den <= num) ++q;
            const unsigned long long kq = q + 1ull;
            lw->slot = sl;
            lw->kp = kq < (unsigned long long)nc ? (int)kq : (int)nc;
            lw->above = run;
          }
        }
        A += mc2;
        run += ns;
      }
    }
    cluster.sync();  // (w2) the boundary is known
    int bslot = lw->slot, bkp = lw->kp;
    if (draw && topp && k_active && bslot < 0) {
      // every top-k survivor is kept: top-k's boundary stands
      bslot = lw->k_slot;
      bkp = lw->k_kept;
    }
    // the best wholly kept regular slot of my range: approximate scores first,
    // then the exact score where it can matter
    float emax = -INFINITY;
    int eslot = -1, etie = 0;
    if (draw) {
      float amax = -INFINITY;
      for (int sl = t0; sl < t1; ++sl) {
        if (sl == tiny || sl == kCatch || (bslot >= 0 && sl >= bslot)) continue;
        const unsigned int na = mc[sl - b0], bbits = mb[sl - b0];
        if (na == 0u || bbits == 0u) continue;
        const float z = zq(sl);
        if (minp && !minp_pass(z, m_t, lmp)) continue;
        amax = fmaxf(amax, approx_score(z, bbits - 1u));
      }
      amax = warp_max(amax);
      if (lane == 0) s.rf[warp] = amax;
      __syncthreads();
      float cmax_a = -INFINITY;
      for (int w = 0; w < kWarps; ++w) cmax_a = fmaxf(cmax_a, s.rf[w]);
      __syncthreads();
      if (cmax_a > -INFINITY) {
        const float margin = 1e-3f * (1.0f + fabsf(cmax_a));
        for (int sl = t0; sl < t1; ++sl) {
          if (sl == tiny || sl == kCatch || (bslot >= 0 && sl >= bslot)) continue;
          const unsigned int na = mc[sl - b0], bbits = mb[sl - b0];
          if (na == 0u || bbits == 0u) continue;
          const float z = zq(sl);
          if (minp && !minp_pass(z, m_t, lmp)) continue;
          if (approx_score(z, bbits - 1u) < cmax_a - margin) continue;
          const float sc = gumbel_score_inl(z, bbits - 1u);
          if (sc > emax) {
            emax = sc;
            eslot = sl;
            etie = 0;
          } else if (sc == emax) {
            etie = 1;
          }
        }
      }
      // CTA best; equal scores of different slots mark a tie
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float e2 = __shfl_xor_sync(0xffffffffu, emax, o);
        const int s2 = __shfl_xor_sync(0xffffffffu, eslot, o);
        const int t2 = __shfl_xor_sync(0xffffffffu, etie, o);
        if (e2 > emax) {
          emax = e2;
          eslot = s2;
          etie = t2;
        } else if (e2 == emax && e2 > -INFINITY && s2 != eslot) {
          etie = 1;
        } else if (e2 == emax) {
          etie |= t2;
        }
      }
      if (lane == 0) {
        s.rf[warp] = emax;
        s.ri[warp] = eslot;
        s.ri[kWarps + warp] = etie;
      }
      __syncthreads();
      if (tid == 0) {
        float e = -INFINITY;
        int es = -1, et = 0;
        for (int w = 0; w < kWarps; ++w) {
          if (s.rf[w] > e) {
            e = s.rf[w];
            es = s.ri[w];
            et = s.ri[kWarps + w];
          } else if (s.rf[w] == e && e > -INFINITY && (s.ri[w] != es || s.ri[kWarps + w])) {
            et = 1;
          }
        }
        s.part.best_score = e;
        s.part.best_slot = es;
        s.part.best_tie = et;
        s.part.best_bits = es >= 0 ? mb[es - b0] : 0u;
      }
    }
    cluster.sync();  // (w3) range bests visible
    VT_CTRACE(c, 13);
    const int fallback = lw->fallback;
    const int nslot = lw->slot_n;
    const unsigned long long above = lw->above;
    float wscore = -INFINITY;
    int wslot = -1;
    unsigned int wbits = 0u;
    int wtie = 0;
    if (draw) {
      for (int r = 0; r < C; ++r) {
        const Part* pr = cluster.map_shared_rank(&s.part, r);
        if (pr->best_score > wscore) {
          wscore = pr->best_score;
          wslot = pr->best_slot;
          wbits = pr->best_bits;
          wtie = pr->best_tie;
        } else if (pr->best_score == wscore && wscore > -INFINITY) {
          wtie = 1;
        }
      }
    }
    const int sp_kept0 = tiny >= 0 && (bslot < 0 || tiny < bslot);
    const int sp_kept1 = bslot < 0;
    const int lslot = last_slot;
    const bool give_up = fallback || wtie ||
                         (draw && bslot < 0 && (lslot == tiny || lslot == kCatch)) ||
                         (want_topn && tot_all < (unsigned long long)n);
    __syncthreads();
    if (give_up) {
      cluster.sync();  // nobody reads another CTA's walk data after this
      return false;
    }

    // ---- pass 2: gather the boundary slot's indices and the top-n keys into the
    // leader; find the winning slot's best element and the last survivor ----------
    VT_CTRACE(c, 9);
    unsigned long long kbest = 0ull;  // filled by the leader from the gathered indices
    int last_j = -1, lastslot_j = -1, cand_j = INT_MAX;
    uint64_t* lg = cluster.map_shared_rank(c.buf, 0);
    int* lcount = cluster.map_shared_rank(&s.gcount, 0);
    uint64_t* lbnd = cluster.map_shared_rank(reinterpret_cast<uint64_t*>(code_mem), 0);
    int* lbcount = cluster.map_shared_rank(&s.gcount2, 0);
    const bool gather_b = draw && bslot >= 0;
    const int bsel = gather_b ? bslot : -2;  // -2 matches nothing
    const int nsel = want_topn ? nslot : -2;
    // A regular slot holds one bf16 value, so the matches are on the raw bits:
    // the boundary, winning and last slots by equality, the top-n slots by
    // order (every value at least the value of slot nsel).  A slot that is
    // not regular matches nothing (the last slot is then unused, and a top-n
    // or boundary slot never is one here).
    auto slot_bits = [&](int sl) -> uint32_t {
      if (sl < 0 || sl == tiny || sl >= kCatch) return 0xFFFFu;  // a NaN: matches no element
      const int code = cmax - sl;
      const uint32_t mag = (uint32_t)((code < 0 ? -code : code) - 1 + (kCodeEmin << 7));
      return (code < 0 ? 0x8000u : 0u) | mag;
    };
    auto ord16 = [](uint32_t u) -> uint32_t { return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u); };
    const uint32_t ub = slot_bits(bsel), uw = slot_bits(wslot), ul = slot_bits(lslot);
    const uint32_t un = slot_bits(nsel);
    const uint32_t kn = un == 0xFFFFu ? 0x10000u : ord16(un);  // 0x10000: no top-n
    // the next group's words are loaded while this one is matched
    uint32_t wnext[8];
    if (tid < ngroups_live) group_words(tid, wnext);
    for (int g = tid; g < ngroups_live; g += kThreads) {
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) w[q] = wnext[q];
      if (g + kThreads < ngroups_live) group_words(g + kThreads, wnext);
      const int j0 = lo + g * 16;
      // match masks of the 16 elements first (no branches), then the rare work
      // (-inf, and the -inf padding past the row end, match nothing)
      unsigned int mb = 0u, mw = 0u, ml = 0u, mn = 0u;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t u = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
        mb |= (u == ub) ? (1u << e) : 0u;
        mw |= (u == uw) ? (1u << e) : 0u;
        ml |= (u == ul) ? (1u << e) : 0u;
        mn |= (ord16(u) >= kn) ? (1u << e) : 0u;
      }
      if ((mb | mw | ml | mn) == 0u) continue;
      if (ml) lastslot_j = max(lastslot_j, j0 + 31 - __clz(ml));
      while (mb) {
        const int e = __ffs(mb) - 1;
        mb &= mb - 1u;
        // descending order of 0xFFFFFFFF - j is ascending index order
        const int pos = atomicAdd(lbcount, 1);
        if (pos < kBufCap) lbnd[pos] = (unsigned long long)(0xFFFFFFFFu - (uint32_t)(j0 + e));
      }
      while (mw) {
        const int e = __ffs(mw) - 1;
        mw &= mw - 1u;
        if (noise_bits(rkey, j0 + e) + 1u == wbits) cand_j = min(cand_j, j0 + e);
      }
      if (mn) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          if ((mn >> e) & 1u) {
            const uint32_t u = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
            const int pos = atomicAdd(lcount, 1);
            if (pos < kBufCap)
              lg[pos] = elem_key(__fmul_rn(__uint_as_float(u << 16), inv_t), (uint32_t)(j0 + e));
          }
        }
      }
    }
    // this CTA's results
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, kbest, o);
      kbest = k2 > kbest ? k2 : kbest;
      last_j = max(last_j, __shfl_xor_sync(0xffffffffu, last_j, o));
      lastslot_j = max(lastslot_j, __shfl_xor_sync(0xffffffffu, lastslot_j, o));
      cand_j = min(cand_j, __shfl_xor_sync(0xffffffffu, cand_j, o));
    }
    if (lane == 0) {
      s.ru[warp] = kbest;
      s.ri[warp] = last_j;
      s.ri[kWarps + warp] = cand_j;
      s.ri[2 * kWarps + warp] = lastslot_j;
    }
    __syncthreads();
    if (tid == 0) {
      unsigned long long kb2 = 0ull;
      int lj = -1, cj = INT_MAX, lsj = -1;
      for (int w = 0; w < kWarps; ++w) {
        kb2 = s.ru[w] > kb2 ? s.ru[w] : kb2;
        lj = max(lj, s.ri[w]);
        cj = min(cj, s.ri[kWarps + w]);
        lsj = max(lsj, s.ri[2 * kWarps + w]);
      }
      s.part.cb_key = kb2;
      s.part.cb_last = lj;
      s.part.cw_j = cj;
      s.part.last_j = lsj;
    }
    VT_CTRACE(c, 14);
    cluster.sync();  // (d) pass-2 parts and top-n keys complete

    // ---- the leader: draw, outputs -------------------------------------------
    if (leader) {
      if (gather_b) {
        // the kept prefix of the boundary slot: its bkp lowest indices
        // (keys 0xFFFFFFFF - j: the bkp largest are the bkp lowest indices)
        uint64_t* bk = reinterpret_cast<uint64_t*>(code_mem);
        const int nbk = min(s.gcount2, kBufCap);
        const int kq = min(bkp, nbk);
        const uint64_t kth = kq >= 1 ? block_select_desc(bk, nbk, kq, s) : ~0ull;
        unsigned long long kb = 0ull;
        for (int t = tid; t < nbk; t += kThreads) {
          if (bk[t] < kth) continue;
          const int j = (int)(0xFFFFFFFFu - (uint32_t)bk[t]);
          const unsigned long long k =
              ((unsigned long long)(noise_bits(rkey, j) + 1u) << 32) | (0xFFFFFFFFu - (uint32_t)j);
          kb = k > kb ? k : kb;
        }
        kb = block_max_u64(kb, s);
        if (tid == 0) {
          s.part.cb_key = kb;
          s.part.cb_last = (bkp >= 1 && bkp <= nbk) ? (int)(0xFFFFFFFFu - (uint32_t)kth) : -1;
          if (s.gcount2 > kBufCap || bkp > nbk) s.part.err |= kErrInternal;
        }
        __syncthreads();
      }
      if (want_topn) {
        const int N = min(s.gcount, kBufCap);
        const int q = min(n, N);
        uint64_t* top = reinterpret_cast<uint64_t*>(s.tmax);
        if (q > 0) block_top_desc(c.buf, N, q, top, s);
        int32_t* out_ids = a.out_topk_ids + (int64_t)row * n;
        float* out_lps = a.out_topk_logprobs + (int64_t)row * n;
        for (int t = tid; t < n; t += kThreads) {
          if (t < q) {
            const uint64_t k = top[t];
            out_ids[t] = (int)key_idx(k);
            out_lps[t] = (key_z(k) - m_t) - lnS;
          } else {
            out_ids[t] = -1;
            out_lps[t] = -INFINITY;
          }
        }
      }
      if (tid == 0) {
        int tok = s.rs.bi;
        float ztok = m_t;
        int kept = 1;
        float kth_v = m_t;
        int kth_i = s.rs.bi;
        int er = 0;
        if (draw) {
          unsigned long long cbk = 0ull;
          int cbl = -1, cwj = INT_MAX, lsj = -1;
          cbk = s.part.cb_key;
          cbl = s.part.cb_last;
          for (int r = 0; r < C; ++r) {
            const Part* pr = cluster.map_shared_rank(&s.part, r);
            cwj = min(cwj, pr->cw_j);
            lsj = max(lsj, pr->last_j);
          }
          // candidates: (score, index) and the tempered value when its slot
          // holds one value (else it is read from the logits)
          float bs = -INFINITY, bz = 0.f;
          int bi = INT_MAX;
          bool bz_known = false;
          auto offer = [&](float sc, int j, float zt, bool known) {
            if (j != INT_MAX && pair_better(sc, j, bs, bi)) {
              bs = sc;
              bi = j;
              bz = zt;
              bz_known = known;
            }
          };
          if (wslot >= 0) {
            if (cwj == INT_MAX)
              er |= kErrInternal;  // the winning slot's best element must exist
            else
              offer(wscore, cwj, zq(wslot), true);
          }
          if (bslot >= 0 && cbk != 0ull) {
            const uint32_t bits = (uint32_t)(cbk >> 32) - 1u;
            const float zb = zq_value(cmax, bslot, inv_t);
            offer(gumbel_score(zb, bits), (int)(0xFFFFFFFFu - (uint32_t)cbk), zb, true);
          }
          if (sp_kept0 && sp_k0 != 0ull) offer(key_z(sp_k0), (int)key_idx(sp_k0), 0.f, false);
          if (sp_kept1 && sp_k1 != 0ull) offer(key_z(sp_k1), (int)key_idx(sp_k1), 0.f, false);
          if (bi == INT_MAX) {
            er |= kErrInternal;
            bi = s.rs.bi;
            bz_known = false;
          }
          tok = bi;
          // the winner's tempered value: its slot's value, or from its logit
          ztok = bz_known ? bz
                          : __fmul_rn(Elt<T>::load1(reinterpret_cast<const T*>(c.rowp) + tok), inv_t);
          if (bslot >= 0) {
            kept = (int)(above + (unsigned long long)bkp);
            kth_v = zq_value(cmax, bslot, inv_t);
            kth_i = cbl;
          } else {
            kept = (int)tot_cnt;
            kth_v = zq_value(cmax, lslot, inv_t);
            kth_i = lsj;
          }
        }
        s.bcast_i[0] = tok;
        a.out_tokens[row] = tok;
        if (a.out_logprobs) a.out_logprobs[row] = (ztok - m_t) - lnS;
        a.row_status[row] = kRowOk;
        a.dbg_kth_value[row] = kth_v;
        a.dbg_kth_index[row] = kth_i;
        a.dbg_kept[row] = kept;
        a.seeds[row] += kSeedStep;
        decay_top_p(a, row, tok);
        er |= s.rs.err | s.part.err;
        if (er) atomicOr(a.err_word, er);
      }
    }
    cluster.sync();  // (e) no DSMEM access after this
    if (leader && a.update_counts) {
      __syncthreads();
      append_token(a.hist + (int64_t)row * a.hist_cap, a.hist_len + row, a.hist_cap,
                   s.bcast_i[0], s, a.row_status + row);
    }
    VT_CTRACE(c, 15);
    return true;
  }
}

// ---------------------------------------------------------------------------
// the selection path of one row (every CTA of the cluster calls it)
// ---------------------------------------------------------------------------
// Top-n by selection when the candidates did not hold it, then the kept set by
// radix selection (top-k by count, top-p by mass) and the draw; the leader
// writes the row's outputs.  c.m_t, c.lnS, s.rs.bi are set by the caller.
template <typename T>
__device__ __noinline__ void slow_row(Ctx& c, Smem& s, const SampleArgs& a, cg::cluster_group& cluster,
                         bool topn_done) {
  constexpr int E = Elt<T>::E;
  const int n = a.n_logprobs;
  const bool leader = c.rank == 0;
  int32_t* out_ids = n > 0 ? a.out_topk_ids + (int64_t)c.row * n : nullptr;
  float* out_lps = n > 0 ? a.out_topk_logprobs + (int64_t)c.row * n : nullptr;
  // level-0 bins by bf16 code for bf16 rows whose values are all bf16
  const bool codes = sizeof(T) == 2 && !c.pen;
  if (n > 0 && !topn_done) {
    {
      // rank n-1 of every element (the -inf ones included, by index)
      SelOut so = cluster_select<T>(c, s, cluster, kPredAll, 0ull, false,
                                    (unsigned long long)(n - 1), 0.f, false, codes);
      const unsigned long long kb = so.all ? 0ull : so.kb;
      if (leader && c.tid == 0) s.gcount = 0;
      cluster.sync();
      uint64_t* lg = cluster.map_shared_rank(c.buf, 0);
      int* lcount = cluster.map_shared_rank(&s.gcount, 0);
      const uint32_t kb_hi = (uint32_t)(kb >> 32);
      for_each_elem<T>(
          c, [&](float gz) { return ord_key(gz) >= kb_hi; },
          [&](float zt, int j) {
            const unsigned long long K = elem_key(zt, (uint32_t)j);
            if (K < kb) return;
            const int pos = atomicAdd(lcount, 1);
            if (pos < kBufCap) lg[pos] = K;
          });
      cluster.sync();
      if (leader) {
        const int N = min(s.gcount, kBufCap);
        block_sort_desc(c.buf, N);
        for (int t = c.tid; t < n; t += kThreads) {
          if (t < N) {
            const uint64_t k = c.buf[t];
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
    cluster.sync();
    if (!leader) return;
  } else {
    bool bounded = false, draw_known = false;
    unsigned long long kb = 0ull, win = kNegInfKey;
    if (c.topk || c.topp) {
      unsigned long long kbk = 0ull;
      if (c.topk) {
        SelOut so = cluster_select<T>(c, s, cluster, kPredSurv, 0ull, false,
                                      (unsigned long long)(c.top_k - 1), 0.f, !c.topp, codes);
        if (!so.all) {
          kbk = so.kb;
          bounded = true;
          kb = so.kb;
          kept = (int)so.cnt_incl;
          if (!c.topp && so.draw_ok) {
            draw_known = true;
            win = so.win;
          }
        } else {
          kept = (int)so.total_cnt;
        }
      }
      if (c.topp) {
        SelOut so =
            cluster_select<T>(c, s, cluster, kPredSurv, kbk, true, 0ull, c.top_p, true, codes);
        if (!so.all) {
          bounded = true;
          kb = so.kb;
          kept = (int)so.cnt_incl;
          if (so.draw_ok) {
            draw_known = true;
            win = so.win;
          }
        } else {
          kept = (int)so.total_cnt;
        }
      }
    }
    if (draw_known) {
      // the winner's tempered logit comes from the CTA that owns its index
      const int wi = (int)key_idx(win);
      if (c.tid == 0 && wi >= c.lo && wi < c.hi) {
        const int g = (wi - c.lo) / E;
        float x[E];
        load_group<T>(c, g, x);
        float xv = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i)
          if (c.lo + g * E + i == wi) xv = x[i];
        cluster.map_shared_rank(&s.bcast_f[0], 0)[0] = __fmul_rn(xv, c.inv_t);
      }
      VT_CTRACE(c, 11);
      cluster.sync();  // final: no DSMEM access after this
      if (!leader) {
        VT_CTRACE(c, 15);
        return;
      }
      tok = wi;
      ztok = s.bcast_f[0];
      kth_v = key_z(kb);
      kth_i = (int)key_idx(kb);
    } else {
    // draw pass over the kept elements
    float s_cur = -INFINITY, bz = 0.f;
    int bidx = INT_MAX;
    int cnt = 0;
    unsigned long long kmin = ~0ull;
    const uint32_t kb_hi = (uint32_t)(kb >> 32);
    const bool threshold_row = !bounded;  // kept = every survivor: count it here
    auto kept_elem = [&](float zt, int j) -> bool {
      if (!(zt > -INFINITY) || j >= c.hi) return false;
      if (c.minp && !minp_pass(zt, c.m_t, c.lmp)) return false;
      return !bounded || elem_key(zt, (uint32_t)j) >= kb;
    };
    auto score_elem = [&](float zt, int j, uint32_t b) {
      if (threshold_row) {
        ++cnt;
        const unsigned long long K = elem_key(zt, (uint32_t)j);
        kmin = K < kmin ? K : kmin;
      }
      if (!may_beat(zt, s_cur, b)) return;
      const float sc = gumbel_score(zt, b);
      if (pair_better(sc, j, s_cur, bidx)) {
        s_cur = sc;
        bidx = j;
        bz = zt;
      }
    };
    for_each_group<T>(
        c, [&](float gz) { return gz > -INFINITY && (!bounded || ord_key(gz) >= kb_hi); },
        [&](float* x, int, int j0) {
#pragma unroll
          for (int i = 0; i < E; i += 2) {
            // one SplitMix64 output serves the column pair (j0 + i, j0 + i + 1)
            const float z0 = __fmul_rn(x[i], c.inv_t), z1 = __fmul_rn(x[i + 1], c.inv_t);
            const bool k0 = kept_elem(z0, j0 + i), k1 = kept_elem(z1, j0 + i + 1);
            if (!(k0 || k1)) continue;
            const uint64_t h = pair_hash(c.rkey, j0 + i);
            if (k0) score_elem(z0, j0 + i, bits_even(h));
            if (k1) score_elem(z1, j0 + i + 1, bits_odd(h));
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
    VT_CTRACE(c, 11);
    cluster.sync();  // final: no DSMEM access after this
    if (!leader) {
      VT_CTRACE(c, 15);
      return;
    }
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
  }
  if (c.tid == 0) {
    a.out_tokens[c.row] = tok;
    if (a.out_logprobs) a.out_logprobs[c.row] = (ztok - c.m_t) - c.lnS;
    a.row_status[c.row] = kRowOk;
    a.dbg_kth_value[c.row] = kth_v;
    a.dbg_kth_index[c.row] = kth_i;
    a.dbg_kept[c.row] = kept;
    a.seeds[c.row] += kSeedStep;
    decay_top_p(a, c.row, tok);
    const int er = s.rs.err | s.part.err;
    if (er) atomicOr(a.err_word, er);
  }
  if (a.update_counts) {
    __syncthreads();
    append_token(a.hist + (int64_t)c.row * a.hist_cap, a.hist_len + c.row, a.hist_cap, tok, s,
                 a.row_status + c.row);
  }
  VT_CTRACE(c, 15);
}

// ---------------------------------------------------------------------------
// kernel 2: the rows kernel 1 handed over, one cluster per row at a time
// ---------------------------------------------------------------------------
// Copy this CTA's slice into shared memory, padded with -inf to whole groups,
// and rebuild its group maxima for the selection kernel's slice size.
template <typename T>
__device__ __noinline__ void stage_slice(Ctx& c, uint8_t* stage_mem) {
  constexpr int E = Elt<T>::E;
  T* st = reinterpret_cast<T*>(stage_mem);
  const T neg_inf = sizeof(T) == 4 ? (T)0 : (T)0xFF80u;  // bf16 -inf; f32 below
  const int nvalid = c.hi > c.lo ? c.hi - c.lo : 0;
  const T* src = reinterpret_cast<const T*>(c.rowp) + c.lo;
  constexpr int per_vec = 16 / (int)sizeof(T);
  const int nfull = c.aligned ? nvalid / per_vec : 0;  // whole 16-byte vectors of the row
  const uint4* src4 = reinterpret_cast<const uint4*>(src);
  uint4* st4 = reinterpret_cast<uint4*>(st);
  for (int v0 = c.tid; v0 < nfull; v0 += 4 * kThreads) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * kThreads;
      if (v < nfull) r[u] = __ldg(src4 + v);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * kThreads;
      if (v < nfull) st4[v] = r[u];
    }
  }
  for (int i = nfull * per_vec + c.tid; i < c.slice; i += kThreads) {
    if constexpr (sizeof(T) == 4) {
      st[i] = i < nvalid ? __ldg(src + i) : -INFINITY;
    } else {
      st[i] = i < nvalid ? __ldg(src + i) : neg_inf;
    }
  }
  __syncthreads();
  c.stage = reinterpret_cast<const uint4*>(stage_mem);
  for (int g = c.tid; g < c.ngroups; g += kThreads) {
    float x[E];
    load_group<T>(c, g, x);
    float gm = x[0];
#pragma unroll
    for (int i = 1; i < E; ++i) gm = fmaxf(gm, x[i]);
    c.gmax[g] = bf16_down(gm);
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) select_kernel(const SampleArgs a,
                                                             const SelectPlan p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ Smem s;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int cid = (int)blockIdx.x / C, G = (int)gridDim.x / C;
  // Rows handed over by the streaming kernel (a list and their statistics),
  // or, when a.early is set, the rows a.rows[0, B) whose statistics this
  // kernel takes itself in a first streaming pass over the slice.
  const bool own_stats = a.early != 0;
  const int count = own_stats ? a.B : (int)a.slow_ctl[0];
  for (int i = cid; i < count; i += G) {
    const int row = own_stats ? (a.rows ? a.rows[i] : i) : a.slow_list[i];
    SlowRow rec;
    if (!own_stats) rec = a.slow[row];
    cluster.sync();  // every CTA of the cluster is done with the previous row
    Ctx c;
    const RowParams P = init_row<T>(c, a, dsm, row, C, rank, p.slice, p.off_gmax, p.off_mrg);
    if (a.trace && rank == 0 && (int64_t)row * p.kernel1_cluster < a.trace_ctas)
      c.trace = a.trace + (size_t)row * p.kernel1_cluster * kTraceSlots;
    VT_CTRACE(c, 10);
    if (c.tid == 0) {
      s.part.err = 0;
      s.nloc = 0;
      s.gcount = 0;
      s.rs.err = 0;
    }
    if (own_stats) {
      // the row's statistics: pass A through the bulk-copy ring (in the code
      // slots' region, free until the selection starts), then the cluster's
      VT_CTRACE(c, 0);
      __syncthreads();
      stream_stats<T>(c, s, dsm + p.off_code);
      VT_CTRACE(c, 2);
      cluster.sync();  // every CTA's partials visible
      VT_CTRACE(c, 3);
      cluster_stats(c, s, cluster);
      __syncthreads();
      const int status0 =
          s.rs.nonfinite ? kRowNonfinite : (s.rs.m_t == -INFINITY ? kRowEmpty : kRowOk);
      rec.m_t = s.rs.m_t;
      rec.lnS = s.rs.lnS;
      rec.xmax = s.rs.bv;
      rec.bi_topn = (uint32_t)s.rs.bi | (a.n_logprobs == 0 ? 0x80000000u : 0u);
      cluster.sync();  // every CTA has read the others' partials
      if (status0 != kRowOk) {
        if (rank == 0) write_bad_row(a, s, row, status0);
        continue;
      }
      if (c.tid == 0) atomicOr(&s.part.err, s.rs.err);
    }
    if (c.tid == 0) s.rs.bi = (int)(rec.bi_topn & 0x7FFFFFFFu);
    c.m_t = rec.m_t;
    c.lnS = rec.lnS;
    c.xmax = rec.xmax;
    const int hist_len = a.hist_len[row];
    if (p.pen_smem && (P.flags & kRowPenalty) != 0 && hist_len > 0)
      setup_penalties<T>(c, s, a, P, dsm, p.off_bitmap, p.off_prefix, hist_len);
    VT_CTRACE(c, 5);
    // bf16 rows without penalties take the code selection, from the staged slice
    // or straight from (aligned) global memory; the rest, or a row the code
    // selection gives back, the generic selection over group maxima
    const bool codes = sizeof(T) == 2 && !c.pen && p.off_code != 0u && (p.staged || c.aligned);
    if (p.staged) stage_slice<T>(c, dsm + p.off_stage);
    VT_CTRACE(c, 1);
    const bool topn_done = (rec.bi_topn >> 31) != 0;
    bool done = false;
    if (codes) done = code_row<T>(c, s, a, cluster, topn_done, dsm + p.off_code);
    if (!done) {
      if (!p.staged) {
        for (int g = c.tid; g < c.ngroups; g += kThreads) {
          float x[Elt<T>::E];
          load_group<T>(c, g, x);
          float gm = x[0];
#pragma unroll
          for (int q = 1; q < Elt<T>::E; ++q) gm = fmaxf(gm, x[q]);
          c.gmax[g] = bf16_down(gm);
        }
        __syncthreads();
      }
      slow_row<T>(c, s, a, cluster, topn_done);
    }
  }
  // The last CTA to finish clears the hand-over counters for the next call.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int done = atomicAdd(&a.slow_ctl[1], 1u);
    if (done == gridDim.x - 1) {
      a.slow_ctl[2] = own_stats ? (unsigned int)count : a.slow_ctl[0];  // for vt_debug_last_handover
      a.slow_ctl[0] = 0u;
      a.slow_ctl[1] = 0u;
      __threadfence();
    }
  }
}

// The count-table append on its own (one CTA per row): used when the call
// exports the filtered distribution, which needs the counts the draw saw.
__global__ void __launch_bounds__(kThreads) append_kernel(int2* hist, int32_t* hist_len,
                                                          int32_t cap, const int32_t* tokens,
                                                          int32_t* row_status) {
  __shared__ Smem s;
  const int row = blockIdx.x;
  if (row_status[row] != kRowOk) return;  // uniform over the CTA
  append_token(hist + (int64_t)row * cap, hist_len + row, cap, tokens[row], s, row_status + row);
}

}  // namespace

// ---------------------------------------------------------------------------
// host side: plans and launches
// ---------------------------------------------------------------------------
LaunchPlan plan_layout(int V, int elem_size, int cluster, bool penalties, bool select) {
  LaunchPlan p;
  p.cluster = cluster;
  int slice = (V + cluster - 1) / cluster;
  slice = (slice + 31) & ~31;
  p.slice = slice;
  p.pen_smem = penalties ? 1 : 0;
  const int E = kGroupBytes / elem_size;
  const size_t ngroups = (size_t)slice / E;
  // Streaming kernel: [0, 32 KB) the pass-A bulk-copy ring, later the
  // candidate buffer (16 KB).  Selection kernel: [0, 16 KB) the gather buffer,
  // aliased by the selection histograms (4 x kBins words), then the merged
  // bins of this CTA's digit range.
  size_t off = select ? (size_t)kBufCap * 8 : (size_t)kRingBytes;
  p.off_gmax = (uint32_t)off;
  off += (ngroups * 2 + 15) & ~(size_t)15;
  p.off_mrg = (uint32_t)off;
  if (select) off += (size_t)(kCodeSlots / cluster) * 12;
  off = (off + 15) & ~(size_t)15;
  p.off_bitmap = (uint32_t)off;
  p.off_prefix = (uint32_t)off;
  if (penalties) {
    off += (size_t)(slice / 32) * 4;
    p.off_prefix = (uint32_t)off;
    off += (size_t)(slice / 32) * 2;
    off = (off + 15) & ~(size_t)15;
    off += (size_t)kSideSmem * 4;  // the slice's penalised values, when they fit
  }
  p.smem = off;
  p.active_clusters = 0;
  p.sel = SelectPlan{};
  return p;
}

// The selection kernel's layout: kernel 1's regions for its own slice size,
// then (when staged) the slice itself.
static SelectPlan plan_select_layout(int V, int elem_size, int cluster, bool penalties,
                                     bool staged) {
  const LaunchPlan q = plan_layout(V, elem_size, cluster, penalties, true);
  SelectPlan p{};
  p.cluster = cluster;
  p.slice = q.slice;
  p.pen_smem = q.pen_smem;
  p.off_gmax = q.off_gmax;
  p.off_mrg = q.off_mrg;
  p.off_bitmap = q.off_bitmap;
  p.off_prefix = q.off_prefix;
  size_t off = (q.smem + 127) & ~(size_t)127;
  p.off_code = 0u;
  if (elem_size == 2) {  // bf16 code slots: counts and best noise bits
    p.off_code = (uint32_t)off;
    // the code slots' counts and best noise bits; the own-statistics pass runs
    // its bulk-copy ring in the same region before the selection starts
    off += (size_t)(kCodeSlots * 8 > kRingBytes ? kCodeSlots * 8 : kRingBytes);
  }
  p.off_stage = (uint32_t)off;
  p.staged = staged ? 1 : 0;
  if (staged) off += (size_t)q.slice * elem_size;
  p.smem = off;
  return p;
}

template <typename T>
static cudaError_t prepare_one(LaunchPlan& plan) {
  // The dynamic shared-memory limit only ever grows, so that every cached
  // plan stays launchable; clusters above 8 CTAs are always allowed.
  static size_t smem_set = 0;
  cudaError_t e = cudaSuccess;
  if (plan.smem > smem_set) {
    e = cudaFuncSetAttribute(sample_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)plan.smem);
    if (e != cudaSuccess) return e;
    smem_set = plan.smem;
  }
  e = cudaFuncSetAttribute(sample_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
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
  int nclusters = 0;
  e = cudaOccupancyMaxActiveClusters(&nclusters, sample_kernel<T>, &cfg);
  if (e != cudaSuccess) return e;
  plan.active_clusters = nclusters;
  return nclusters > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <typename T>
static cudaLaunchConfig_t select_config(const SelectPlan& plan, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Kernel attributes of the selection kernel; plan.clusters = how many of its
// clusters are resident at once.
template <typename T>
static cudaError_t prepare_select_one(SelectPlan& plan) {
  static size_t smem_set = 0;
  cudaError_t e = cudaSuccess;
  if (plan.smem > smem_set) {
    e = cudaFuncSetAttribute(select_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)plan.smem);
    if (e != cudaSuccess) return e;
    smem_set = plan.smem;
  }
  e = cudaFuncSetAttribute(select_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = select_config<T>(plan, attr);
  int nclusters = 0;
  e = cudaOccupancyMaxActiveClusters(&nclusters, select_kernel<T>, &cfg);
  if (e != cudaSuccess) return e;
  plan.clusters = nclusters;
  return nclusters > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t prepare_sample(LaunchPlan& plan, int dtype) {
  cudaError_t e = dtype == 0 ? prepare_one<float>(plan) : prepare_one<uint16_t>(plan);
  if (e != cudaSuccess || plan.sel.cluster == 0) return e;
  const int want = plan.sel.clusters;
  e = dtype == 0 ? prepare_select_one<float>(plan.sel) : prepare_select_one<uint16_t>(plan.sel);
  if (want > 0 && want < plan.sel.clusters) plan.sel.clusters = want;
  return e;
}

// The selection kernel: CTAs per row such that a slice holds at least 16K
// elements (fewer, fuller CTAs keep the cluster barriers cheap), more while
// a slice is over 96 KB; staged in shared memory when it fits in 96 KB; as
// many persistent clusters as are resident at once, at most one per row.
static SelectPlan plan_select(int B, int V, int elem_size, bool penalties, int dtype,
                              int kernel1_cluster) {
  int C = kMaxCluster;
  bool staged;
  if (elem_size == 2) {
    // bf16: the code selection reads each slice twice from global memory, so
    // no staging; slices of at least 32K elements keep the cluster small and
    // many clusters resident
    while (C > 1 && (V + C - 1) / C < 32768) C >>= 1;
    staged = false;
  } else {
    while (C > 1 && (V + C - 1) / C < 16384) C >>= 1;
    while (C < kMaxCluster && (size_t)((V + C - 1) / C) * elem_size > 96 * 1024) C <<= 1;
    staged = (size_t)((V + C - 1) / C + 31) * elem_size <= 96 * 1024;
  }
  SelectPlan p = plan_select_layout(V, elem_size, C, penalties, staged);
  p.kernel1_cluster = kernel1_cluster;
  const cudaError_t e = dtype == 0 ? prepare_select_one<float>(p) : prepare_select_one<uint16_t>(p);
  if (e != cudaSuccess) {
    p.clusters = 0;
    return p;
  }
  if (p.clusters > B) p.clusters = B;
  return p;
}

// The selection kernel that takes its rows' statistics itself (bf16 rows
// without penalties): the streaming kernel's cluster, so that its slices, and
// the statistics summed over them, are the streaming kernel's exactly.
static SelectPlan plan_select_own(int V, int elem_size, int dtype, const LaunchPlan& k1) {
  SelectPlan p{};
  if (elem_size != 2 || dtype == 0) return p;
  p = plan_select_layout(V, elem_size, k1.cluster, false, false);
  p.kernel1_cluster = k1.cluster;
  if (p.off_code == 0u || p.slice != k1.slice ||
      prepare_select_one<uint16_t>(p) != cudaSuccess) {
    SelectPlan none{};
    return none;
  }
  return p;
}

LaunchPlan plan_sample(int B, int V, int elem_size, bool penalties, int dtype, int num_sms) {
  // Slices of at most 512 KB (so the per-group structures stay small) and at
  // least 8 KB of logits; among those, the largest cluster that still lets
  // all B rows be resident at once, else the smallest one.
  (void)num_sms;
  const size_t max_slice = 512 * 1024, min_slice = 8 * 1024;
  int cmin = 1;
  while (cmin < kMaxCluster && (size_t)((V + cmin - 1) / cmin) * elem_size > max_slice) cmin <<= 1;
  LaunchPlan best = plan_layout(V, elem_size, cmin, penalties, false);
  if (prepare_sample(best, dtype) != cudaSuccess) return best;
  if ((int64_t)B > best.active_clusters) {  // several waves even so
    best.sel = plan_select(B, V, elem_size, penalties, dtype, best.cluster);
    best.own = plan_select_own(V, elem_size, dtype, best);
    return best;
  }
  for (int C = cmin * 2; C <= kMaxCluster; C <<= 1) {
    if ((size_t)((V + C - 1) / C) * elem_size < min_slice) break;
    LaunchPlan p = plan_layout(V, elem_size, C, penalties, false);
    if (prepare_sample(p, dtype) != cudaSuccess) break;
    if ((int64_t)B > p.active_clusters) break;  // would no longer fit in one wave
    best = p;
  }
  best.sel = plan_select(B, V, elem_size, penalties, dtype, best.cluster);
  best.own = plan_select_own(V, elem_size, dtype, best);
  return best;
}

template <typename T>
static cudaError_t launch_one(const SampleArgs& args, const LaunchPlan& plan,
                              cudaStream_t stream, cudaEvent_t between) {
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, sample_kernel<T>, args);
  if (e != cudaSuccess) return e;
  if (between) {
    e = cudaEventRecord(between, stream);
    if (e != cudaSuccess) return e;
  }
  if (plan.sel.clusters < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t cfg2 = select_config<T>(plan.sel, attr2);
  cfg2.gridDim = dim3((unsigned)(plan.sel.clusters * plan.sel.cluster), 1, 1);
  cfg2.stream = stream;
  return cudaLaunchKernelEx(&cfg2, select_kernel<T>, args, plan.sel);
}

cudaError_t launch_sample(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                          cudaStream_t stream, cudaEvent_t between) {
  return dtype == 0 ? launch_one<float>(args, plan, stream, between)
                    : launch_one<uint16_t>(args, plan, stream, between);
}

cudaError_t launch_select_handed(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                                 cudaStream_t stream, int max_clusters) {
  if (plan.sel.clusters < 1) return cudaErrorInvalidConfiguration;
  const int G = (max_clusters > 0 && max_clusters < plan.sel.clusters) ? max_clusters
                                                                      : plan.sel.clusters;
  cudaLaunchAttribute attr[1];
  if (dtype == 0) {
    cudaLaunchConfig_t cfg = select_config<float>(plan.sel, attr);
    cfg.gridDim = dim3((unsigned)(G * plan.sel.cluster), 1, 1);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, select_kernel<float>, args, plan.sel);
  }
  cudaLaunchConfig_t cfg = select_config<uint16_t>(plan.sel, attr);
  cfg.gridDim = dim3((unsigned)(G * plan.sel.cluster), 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, select_kernel<uint16_t>, args, plan.sel);
}

cudaError_t launch_select_own(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                              cudaStream_t stream, cudaEvent_t launched) {
  if (dtype == 0 || plan.own.cluster < 1 || !args.early) return cudaErrorInvalidValue;
  if (args.B < 1) return launched ? cudaEventRecord(launched, stream) : cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = select_config<uint16_t>(plan.own, attr);
  cfg.gridDim = dim3((unsigned)(args.B * plan.own.cluster), 1, 1);
  cfg.stream = stream;
  if (launched) {  // fires once every CTA of the launch has begun
    attr[1].id = cudaLaunchAttributeLaunchCompletionEvent;
    attr[1].val.launchCompletionEvent.event = launched;
    attr[1].val.launchCompletionEvent.flags = 0;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, select_kernel<uint16_t>, args, plan.own);
}

namespace {
// A wait that nothing completes (an mbarrier expecting one arrival that never
// comes), bounded by `limit_ns`: the kernel records kErrTimeout and returns,
// as every bounded wait of the sampling kernels does when it runs out.
__global__ void wait_probe_kernel(int32_t* err_word, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait_bounded(&bar, 0u, limit_ns)) atomicOr(err_word, kErrTimeout);
}
}  // namespace

cudaError_t launch_wait_probe(int32_t* err_word, unsigned long long limit_ns,
                              cudaStream_t stream) {
  wait_probe_kernel<<<1, 1, 0, stream>>>(err_word, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_append(int2* hist, int32_t* hist_len, int32_t hist_cap, const int32_t* tokens,
                          int32_t* row_status, int B, cudaStream_t stream) {
  if (B < 1) return cudaSuccess;
  append_kernel<<<B, kThreads, 0, stream>>>(hist, hist_len, hist_cap, tokens, row_status);
  return cudaGetLastError();
}

}  // namespace vt
