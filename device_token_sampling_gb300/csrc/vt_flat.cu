// vt_flat.cu -- the flat kernels: bf16 batches without penalties or top-p decay.
//
// The row pipeline of the pages (temperature, min-p, top-k, top-p over the
// survivors renormalised, the seeded Gumbel-max draw with lowest-index ties,
// log-probs and top-n) in six launches over (row, slice) pairs, none of whose
// CTAs waits on another:
//
//   P1 stats    (row, slice): the slice is read once from HBM into registers;
//               its maximum, lowest-index argmax and sum of exp(z_t - m) (the
//               log-softmax statistics of the pages), and every thread's
//               maximum (a bf16 code) for the row's candidate threshold.
//   P2 row      (row): the row's statistics; its route; the candidate
//               threshold tau, the K-th largest of the C x 256 thread maxima
//               (at least K elements are >= tau, K = max(top_k, n)); for rows
//               without top-k the Gumbel score of the row's maximum; for
//               top-p rows, per code slot, its mass and the noise bits from
//               which one of its elements may out-score the maximum, and the
//               first slot that holds no survivor.
//   P2 -> P3 the slices are read again (from L2):
//   P3 collect  (row, slice): the elements >= tau as candidate keys; for rows
//               without top-k the survivors' count and last key, the draw
//               contenders (elements whose Gumbel score beats the maximum's:
//               the winner is one of them or the maximum itself), and for
//               top-p rows a count per bf16 code slot, summed into 64 coarse
//               bins of exact 2^-43 fixed-point masses.
//   P4 finish   (row): top-n from the candidates (sorted when few, else
//               selected then sorted); rows with top-k (or
//               greedy) settle on the candidates exactly as on the whole row;
//               rows without top-p settle on the survivors and contenders;
//               top-p rows find the coarse bin holding the nucleus boundary.
//   P5 fine     (row, slice), top-p rows: counts per code slot of that bin.
//   P6 top-p    (row): the boundary slot and the kept count inside it (its
//               elements share one mass), the boundary element (the t-th of
//               the slot in index order), and the winner among the kept
//               contenders.
//
// A row the launches cannot settle exactly (a top_k above kFlatKMax, more
// candidates or contenders than their buffers hold, a boundary inside the
// code slot that merges the magnitudes below 2^-12 or in the catch-all) is
// handed to the selection kernel through its SlowRow record, with the
// statistics P2 computed; the flat kernels then write none of its outputs
// except, when P4 wrote them, its top-n.
#include "vt_device.cuh"
#include "vt_kernels.h"

#include <cuda_bf16.h>

#include <climits>
#include <cstring>

namespace vt {
namespace {

constexpr int kFT = 256;            // threads of the per-slice kernels
constexpr int kFW = kFT / 32;
constexpr int kFF = 512;            // threads of the per-row statistics kernel
constexpr int kF4 = 256;            // threads of the per-row completion kernel
constexpr int kSmallCand = 256;     // candidates the completion kernel sorts outright
constexpr int kSliceCand = 1024;    // candidate keys one slice CTA stages
constexpr int kSliceCont = 128;     // contenders one slice CTA stages
constexpr int kTinySlotNone = -1;
constexpr int kFlatSlice = 9728;    // elements per slice at most (5 vectors a thread)
constexpr float kGumbelMax = 17.5f; // above -ln(-ln(1 - 2^-25)) = 17.33, the largest noise

// Row routes.
enum : int32_t {
  kRouteDone = 0,   // outputs written (or a bad row)
  kRouteHand = 1,   // handed to the selection kernel
  kRouteCand = 2,   // settled on the candidates (greedy, or 1 < top_k <= kFlatKMax)
  kRouteHist = 3,   // no top-k: survivors, contenders, and for top-p the code slots
  kRouteFine = 4,   // top-p row after P4: the boundary bin is known
};

// P1 -> P2, per (row, slice).
struct __align__(16) FlatSlice {
  float m_t;        // tempered maximum of the slice (-inf: none finite)
  float s;          // sum of exp(z_t - m_t) over the slice
  int32_t argj;     // lowest index of the maximum (INT_MAX: none)
  uint32_t flags;   // bit 0: a NaN seen; bits 16..31: the maximum's bf16 bits
};

// Per row, written by P2 and read by the later launches.
struct __align__(16) FlatRow {
  float m_t, lnS;
  int32_t argj;
  int32_t route;
  float tau_x;                 // candidates: x >= tau_x (+inf: none)
  int32_t cmax;                // code16 of the maximum
  float score_top;             // Gumbel score of the maximum
  int32_t dcut;                // top-p rows: regular slots >= dcut hold no survivor of mass > 0
  int32_t tiny;                // the slot of code 0, or kTinySlotNone
  uint32_t ncand;              // candidates appended
  uint32_t ncont;              // contenders appended
  uint32_t overflow;           // a buffer overflowed: hand over
  uint32_t surv;               // rows without top-p: survivors
  int32_t bstar;               // top-p rows: the boundary's coarse bin
  unsigned long long lastkey;  // rows without top-p: smallest survivor key (as ~key, max)
  unsigned long long tm;       // floor(W p)
  unsigned long long above;    // mass of the bins before bstar
  uint32_t cabove;             // elements in the bins before bstar
  uint32_t tau16;              // ord16 code of tau_x (0x10000: no candidates)
};

// P3 -> P4/P6, per (row, slice) of top-p rows.
struct __align__(16) FlatHist {
  unsigned long long mass[kFlatBins];
  uint32_t cnt[kFlatBins];
  unsigned long long tiny_mass, catch_mass;
  uint32_t tiny_cnt, catch_cnt;
};

struct __align__(16) Contender {
  float score;
  int32_t j;
  float z;
  int32_t d;   // code slot (top-p rows)
};

// Scratch carving (every region 256-byte aligned).
struct FlatMem {
  FlatSlice* slices;   // [B][C]
  uint16_t* tmax;      // [B][C][kFT]
  FlatRow* rows;       // [B]
  uint64_t* cand;      // [B][kFlatCandCap]
  Contender* cont;     // [B][kFlatContCap]
  FlatHist* hist;      // [B][C]
  uint32_t* fine;      // [B][C][kFlatBins]
  unsigned long long* wtab;  // [B][kCodeSlots] top-p rows: each survivor slot's mass
  uint32_t* btab;      // [B][kCodeSlots] top-p rows: noise bits from which a slot's
                       // element may out-score the maximum (2^24: never)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline FlatMem carve(void* base, int B, int C) {
  FlatMem m;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  m.slices = reinterpret_cast<FlatSlice*>(p + off);
  off = align256(off + sizeof(FlatSlice) * (size_t)B * C);
  m.tmax = reinterpret_cast<uint16_t*>(p + off);
  off = align256(off + sizeof(uint16_t) * (size_t)B * C * kFT);
  m.rows = reinterpret_cast<FlatRow*>(p + off);
  off = align256(off + sizeof(FlatRow) * (size_t)B);
  m.cand = reinterpret_cast<uint64_t*>(p + off);
  off = align256(off + sizeof(uint64_t) * (size_t)B * kFlatCandCap);
  m.cont = reinterpret_cast<Contender*>(p + off);
  off = align256(off + sizeof(Contender) * (size_t)B * kFlatContCap);
  m.hist = reinterpret_cast<FlatHist*>(p + off);
  off = align256(off + sizeof(FlatHist) * (size_t)B * C);
  m.fine = reinterpret_cast<uint32_t*>(p + off);
  off = align256(off + sizeof(uint32_t) * (size_t)B * C * kFlatBins);
  m.wtab = reinterpret_cast<unsigned long long*>(p + off);
  off = align256(off + sizeof(unsigned long long) * (size_t)B * kCodeSlots);
  m.btab = reinterpret_cast<uint32_t*>(p + off);
  return m;
}

__host__ __device__ inline size_t carve_bytes(int B, int C) {
  size_t off = 0;
  off = align256(off + sizeof(FlatSlice) * (size_t)B * C);
  off = align256(off + sizeof(uint16_t) * (size_t)B * C * kFT);
  off = align256(off + sizeof(FlatRow) * (size_t)B);
  off = align256(off + sizeof(uint64_t) * (size_t)B * kFlatCandCap);
  off = align256(off + sizeof(Contender) * (size_t)B * kFlatContCap);
  off = align256(off + sizeof(FlatHist) * (size_t)B * C);
  off = align256(off + sizeof(uint32_t) * (size_t)B * C * kFlatBins);
  off = align256(off + sizeof(unsigned long long) * (size_t)B * kCodeSlots);
  off = align256(off + sizeof(uint32_t) * (size_t)B * kCodeSlots);
  return off;
}

// Order-preserving 16-bit code of a bf16 pattern (larger code, larger value;
// both zeros as +0).  NaN patterns are not passed in.
__device__ __forceinline__ uint32_t ord16(uint32_t u) {
  u &= 0xFFFFu;
  if (u == 0x8000u) u = 0u;
  return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
}
__device__ __forceinline__ float ord16_value(uint32_t o) {
  const uint32_t u = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  return __uint_as_float(u << 16);
}

// Element e (0..7) of a vector of 8 bf16: the bit pattern and the value.
__device__ __forceinline__ uint32_t bits_of(const uint4& v, int e) {
  const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}
__device__ __forceinline__ float val_of(const uint4& v, int e) {
  const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// Vector c of the slice [lo, hi) of row x: 8 bf16, -inf past hi (16-byte
// aligned rows; only the row's last vector can be partial).
__device__ __forceinline__ uint4 load_vec(const uint16_t* x, int lo, int hi, int c) {
  const int j0 = lo + 8 * c;
  if (j0 + 8 <= hi) return __ldg(reinterpret_cast<const uint4*>(x + j0));
  uint32_t h[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) h[e] = j0 + e < hi ? (uint32_t)__ldg(x + j0 + e) : 0xFF80u;
  return make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
}

constexpr uint32_t kNegInf2 = 0xFF80FF80u;

// Largest of the 8 bf16 of a vector, NaN when any of them is NaN.
__device__ __forceinline__ float vec_max(const uint4& v) {
  __nv_bfloat162 h[4];
  memcpy(&h[0], &v.x, 4);
  memcpy(&h[1], &v.y, 4);
  memcpy(&h[2], &v.z, 4);
  memcpy(&h[3], &v.w, 4);
  const __nv_bfloat162 a = __hmax2_nan(__hmax2_nan(h[0], h[1]), __hmax2_nan(h[2], h[3]));
  return __bfloat162float(__hmax_nan(__low2bfloat16(a), __high2bfloat16(a)));
}

// Block reductions over the NT threads of a CTA (every thread calls; all get
// the result).
struct RedSmem {
  float f[32];
  int i[32];
  unsigned long long u[32];
  float bf, bz;
  int bi;
  unsigned long long bu;
};

template <int NT>
__device__ float bmax_f(float v, RedSmem& r) {
  constexpr int NW = NT / 32;
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) r.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < NW ? r.f[threadIdx.x] : -INFINITY;
    t = warp_max(t);
    if (threadIdx.x == 0) r.bf = t;
  }
  __syncthreads();
  const float out = r.bf;
  __syncthreads();
  return out;
}

template <int NT>
__device__ float bsum_f(float v, RedSmem& r) {
  constexpr int NW = NT / 32;
  v = warp_sum_f(v);
  if ((threadIdx.x & 31) == 0) r.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < NW ? r.f[threadIdx.x] : 0.f;
    t = warp_sum_f(t);
    if (threadIdx.x == 0) r.bf = t;
  }
  __syncthreads();
  const float out = r.bf;
  __syncthreads();
  return out;
}

template <int NT>
__device__ int bmin_i(int v, RedSmem& r) {
  constexpr int NW = NT / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) r.i[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int t = threadIdx.x < NW ? r.i[threadIdx.x] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = min(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (threadIdx.x == 0) r.bi = t;
  }
  __syncthreads();
  const int out = r.bi;
  __syncthreads();
  return out;
}

template <int NT>
__device__ unsigned long long bsum_u64(unsigned long long v, RedSmem& r) {
  constexpr int NW = NT / 32;
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) r.u[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < NW ? r.u[threadIdx.x] : 0ull;
    t = warp_sum_u64(t);
    if (threadIdx.x == 0) r.bu = t;
  }
  __syncthreads();
  const unsigned long long out = r.bu;
  __syncthreads();
  return out;
}

template <int NT>
__device__ unsigned long long bmax_u64(unsigned long long v, RedSmem& r) {
  constexpr int NW = NT / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
    v = t > v ? t : v;
  }
  if ((threadIdx.x & 31) == 0) r.u[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < NW ? r.u[threadIdx.x] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long q = __shfl_xor_sync(0xffffffffu, t, o);
      t = q > t ? q : t;
    }
    if (threadIdx.x == 0) r.bu = t;
  }
  __syncthreads();
  const unsigned long long out = r.bu;
  __syncthreads();
  return out;
}

// Block argmax of (score, index) -- the larger score, then the lower index --
// carrying z along.
template <int NT>
__device__ void bargmax(float& v, int& j, float& z, RedSmem& r) {
  constexpr int NW = NT / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int j2 = __shfl_xor_sync(0xffffffffu, j, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    if (pair_better(v2, j2, v, j)) {
      v = v2;
      j = j2;
      z = z2;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    r.f[warp] = v;
    r.i[warp] = j;
    r.u[warp] = __float_as_uint(z);
  }
  __syncthreads();
  if (warp == 0) {
    float tv = lane < NW ? r.f[lane] : -INFINITY;
    int tj = lane < NW ? r.i[lane] : INT_MAX;
    float tz = lane < NW ? __uint_as_float((uint32_t)r.u[lane]) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, tv, o);
      const int j2 = __shfl_xor_sync(0xffffffffu, tj, o);
      const float z2 = __shfl_xor_sync(0xffffffffu, tz, o);
      if (pair_better(v2, j2, tv, tj)) {
        tv = v2;
        tj = j2;
        tz = z2;
      }
    }
    if (lane == 0) {
      r.bf = tv;
      r.bi = tj;
      r.bz = tz;
    }
  }
  __syncthreads();
  v = r.bf;
  j = r.bi;
  z = r.bz;
  __syncthreads();
}

// Exclusive prefix over the NT threads of one u64 each; *total gets the sum.
template <int NT>
__device__ unsigned long long bexscan_u64(unsigned long long v, unsigned long long* total,
                                          RedSmem& r) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) r.u[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = lane < NW ? r.u[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long q = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += q;
    }
    if (lane < NW) r.u[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const unsigned long long before = warp == 0 ? 0ull : r.u[warp - 1];
  *total = r.u[NW - 1];
  __syncthreads();
  return before + inc - v;
}

// Outputs of a settled row (one thread).
__device__ __forceinline__ void write_row(const FlatArgs& a, int row, int tok, float ztok,
                                          float m_t, float lnS, float kth_z, int kth_j,
                                          int kept) {
  a.out_tokens[row] = tok;
  if (a.out_logprobs) a.out_logprobs[row] = (ztok - m_t) - lnS;
  a.row_status[row] = kRowOk;
  a.dbg_kth_value[row] = kth_z;
  a.dbg_kth_index[row] = kth_j;
  a.dbg_kept[row] = kept;
  a.seeds[row] += kSeedStep;
}

// Hand a row to the selection kernel (one thread); its SlowRow record holds
// the row's statistics already.
__device__ __forceinline__ void hand_over(const FlatArgs& a, FlatRow& R, int row,
                                         bool topn_written) {
  if (topn_written) a.slow[row].bi_topn |= 0x80000000u;
  R.route = kRouteHand;
  const uint32_t i = atomicAdd(&a.slow_ctl[0], 1u);
  a.slow_list[i] = row;
}

// ---------------------------------------------------------------------------
// P1: per-slice statistics (the one read of the logits from HBM)
// ---------------------------------------------------------------------------
template <int NV>
__global__ void __launch_bounds__(kFT) flat_stats_kernel(const FlatArgs a) {
  __shared__ RedSmem red;
  const int sl = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
  const int lo = sl * a.L, hi = min(a.V, lo + a.L);
  const int nvec = (hi - lo + 7) >> 3;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(a.logits) + (int64_t)row * a.ld;
  const FlatMem M = carve(a.scratch, a.B, a.C);
  const float inv_t = a.params[row].inv_t;

  uint4 v[NV];
  float vmax[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = tid + i * kFT;
    v[i] = c < nvec ? load_vec(x, lo, hi, c) : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
  float tmx = -INFINITY;
  bool nan_seen = false;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    vmax[i] = vec_max(v[i]);
    nan_seen |= vmax[i] != vmax[i];
    tmx = fmaxf(tmx, vmax[i]);
  }
  nan_seen = __syncthreads_or(nan_seen) != 0;
  const float xmax = bmax_f<kFT>(tmx, red);
  // the lowest index holding the maximum
  int bj = INT_MAX;
  if (xmax > -INFINITY) {
#pragma unroll
    for (int i = NV - 1; i >= 0; --i) {
      if (vmax[i] == xmax) {
#pragma unroll
        for (int e = 7; e >= 0; --e)
          if (val_of(v[i], e) == xmax) bj = lo + 8 * (tid + i * kFT) + e;
      }
    }
  }
  bj = bmin_i<kFT>(bj, red);
  // sum of exp(z_t - m) against the slice maximum, in the streaming kernel's
  // arithmetic; vectors whose maximum lies more than 46 / (log2(e) / T) below
  // add less than 2^-46 an element and are skipped
  const float m_t = __fmul_rn(xmax, inv_t);
  float sum = 0.f;
  if (xmax > -INFINITY && xmax < INFINITY && !nan_seen) {
    const float ax = inv_t * kLog2e;
    const float nb = -xmax * ax;
    const float xthr = xmax - 46.0f / ax;
    const bool near0 = fabsf(m_t) <= 16.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (vmax[i] >= xthr) {
        float t[8];
        if (near0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = ex2_approx(fmaf(val_of(v[i], e), ax, nb));
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            t[e] = ex2_approx(__fmul_rn(__fsub_rn(__fmul_rn(val_of(v[i], e), inv_t), m_t), kLog2e));
        }
        sum += ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
      }
    }
  }
  sum = bsum_f<kFT>(sum, red);
  M.tmax[((size_t)row * a.C + sl) * kFT + tid] = (uint16_t)ord16(__float_as_uint(tmx) >> 16);
  if (tid == 0) {
    FlatSlice fs;
    fs.m_t = m_t;
    fs.s = sum;
    fs.argj = bj;
    fs.flags = (nan_seen ? 1u : 0u) | (__float_as_uint(xmax) & 0xFFFF0000u);
    M.slices[(size_t)row * a.C + sl] = fs;
  }
}

// ---------------------------------------------------------------------------
// P2: per-row statistics, route and thresholds
// ---------------------------------------------------------------------------
struct RowSmem {
  uint16_t tm[kFlatMaxC * kFT];  // the row's thread maxima
  unsigned int hist[256];
  int bin, rank;
  int dmin;
};

// Of the 16-bit codes vals[0, N), the K-th largest (1 <= K): two passes of a
// 256-bin histogram, high byte then low byte.  Returns -1 when fewer than K
// codes are at least `floor`.
__device__ int kth_code(const uint16_t* vals, int N, int K, uint32_t floor, RowSmem& s) {
  int prefix = 0;
  int r = K;
  for (int pass = 0; pass < 2; ++pass) {
    for (int b = threadIdx.x; b < 256; b += kFF) s.hist[b] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += kFF) {
      const uint32_t c = vals[i];
      if (c < floor) continue;
      if (pass == 0)
        atomicAdd(&s.hist[c >> 8], 1u);
      else if ((int)(c >> 8) == prefix)
        atomicAdd(&s.hist[c & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bin_desc(s.hist, r, &s.bin, &s.rank);
    __syncthreads();
    if (s.bin < 0) return -1;
    prefix = pass == 0 ? s.bin : ((prefix << 8) | s.bin);
    r = s.rank;
    __syncthreads();
  }
  return prefix;
}

__global__ void __launch_bounds__(kFF) flat_row_kernel(const FlatArgs a) {
  __shared__ RowSmem s;
  __shared__ float sh_m, sh_s;
  __shared__ int sh_argj, sh_bad;
  __shared__ uint32_t sh_xbits;
  const int row = blockIdx.x, tid = threadIdx.x;
  const FlatMem M = carve(a.scratch, a.B, a.C);
  FlatRow& R = M.rows[row];
  const RowParams P = a.params[row];
  const int n = a.n_logprobs;
  if (tid < 32) {
    float m = -INFINITY, sm = 0.f;
    int j = INT_MAX;
    uint32_t xo = 0u, bad = 0u;  // xo: ord16 of the maximum's bits
    if (tid < a.C) {
      const FlatSlice fs = M.slices[(size_t)row * a.C + tid];
      m = fs.m_t;
      sm = fs.s;
      j = fs.argj;
      bad = fs.flags & 1u;
      const uint32_t xb = fs.flags >> 16;
      bad |= (xb == 0x7F80u) ? 1u : 0u;  // +inf
      xo = fs.argj == INT_MAX ? 0u : ord16(xb);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
      const uint32_t xo2 = __shfl_xor_sync(0xffffffffu, xo, o);
      const int j2 = __shfl_xor_sync(0xffffffffu, j, o);
      lse_combine(m, sm, m2, s2, kLog2e);
      if (xo2 > xo || (xo2 == xo && j2 < j)) {
        xo = xo2;
        j = j2;
      }
    }
    bad = __any_sync(0xffffffffu, bad != 0u) ? 1u : 0u;
    if (tid == 0) {
      sh_m = m;
      sh_s = sm;
      sh_argj = j;
      sh_bad = (int)bad;
      sh_xbits = j == INT_MAX ? 0xFF80u : ((xo & 0x8000u) ? (xo & 0x7FFFu) : (~xo & 0xFFFFu));
    }
  }
  __syncthreads();
  const float m_t = sh_m;
  const float lnS = logf(sh_s);
  const int argj = sh_argj;
  const uint32_t xbits = sh_xbits;
  const int status = sh_bad ? kRowNonfinite : (m_t == -INFINITY ? kRowEmpty : kRowOk);
  if (status != kRowOk) {
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
      R.route = kRouteDone;
    }
    return;
  }
  const bool greedy = (P.flags & kRowGreedy) != 0;
  const bool topk = !greedy && P.top_k > 1 && P.top_k < a.V;
  if (tid == 0) {
    SlowRow rec;
    rec.m_t = m_t;
    rec.lnS = lnS;
    rec.xmax = __uint_as_float(xbits << 16);
    rec.bi_topn = (uint32_t)argj | (n == 0 ? 0x80000000u : 0u);
    a.slow[row] = rec;
    R.m_t = m_t;
    R.lnS = lnS;
    R.argj = argj;
    R.ncand = 0u;
    R.ncont = 0u;
    R.overflow = 0u;
    R.surv = 0u;
    R.lastkey = 0ull;
  }
  if (greedy && n == 0) {  // nothing but the argmax
    if (tid == 0) {
      write_row(a, row, argj, m_t, m_t, lnS, m_t, argj, 1);
      R.route = kRouteDone;
    }
    return;
  }
  if (topk && P.top_k > kFlatKMax) {
    if (tid == 0) hand_over(a, R, row, false);
    return;
  }
  // the candidate threshold: the K-th largest thread maximum
  const int K = topk ? max(P.top_k, n) : (greedy ? max(n, 1) : n);
  float tau_x = INFINITY;
  uint32_t tau16 = 0x10000u;
  if (K > 0) {
    const uint16_t* tsrc = M.tmax + (size_t)row * a.C * kFT;
    for (int i = tid; i < a.C * kFT; i += kFF) s.tm[i] = tsrc[i];
    __syncthreads();
    const int code = kth_code(s.tm, a.C * kFT, K, 0x0080u, s);
    if (code < 0) {  // fewer than K thread maxima are finite
      if (tid == 0) hand_over(a, R, row, false);
      return;
    }
    tau_x = ord16_value((uint32_t)code);
    tau16 = (uint32_t)code;
  }
  if (greedy || topk) {
    if (tid == 0) {
      R.tau_x = tau_x;
      R.tau16 = tau16;
      R.route = kRouteCand;
    }
    return;
  }
  // rows without top-k: the maximum's Gumbel score, its code and, for top-p
  // rows, the first regular code slot without survivors of mass > 0
  const int cmax = code16(xbits);
  const int tiny = (cmax >= 0 && cmax < kCodeSlots - 1) ? cmax : kTinySlotNone;
  const bool topp = (P.flags & kRowTopP) != 0;
  const bool minp = (P.flags & kRowMinP) != 0;
  const float score_top = gumbel_score(m_t, noise_bits(row_key(a.seeds[row], row), argj));
  if (tid == 0) s.dmin = kCodeSlots - 1;
  __syncthreads();
  if (topp) {
    // per regular slot: its mass (0: no survivor), and the noise bits b from
    // which the certificate -ln u >= 1 - u no longer rules out a score above
    // the maximum's: with 1 - u = (2^25 - 2b - 1) 2^-25 and t = exp(z_t -
    // score) (expf within 2 ulp, a 2^-7 margin), b <= (2^25 - 1 - T) >> 1 with
    // T = ceil(t 2^25) is ruled out
    unsigned long long* wt = M.wtab + (size_t)row * kCodeSlots;
    uint32_t* bt = M.btab + (size_t)row * kCodeSlots;
    int dm = kCodeSlots - 1;
    for (int d = tid; d < kCodeSlots; d += kFF) {
      unsigned long long w = 0ull;
      uint32_t bmin = 1u << 24;
      if (d != tiny && d < kCodeSlots - 1) {
        const int code = cmax - d;
        bool fail = code < -17920;  // below the most negative finite bf16
        if (!fail) {
          const float z = __fmul_rn(code_value(code), P.inv_t);
          w = mass_fixed(z, m_t);
          fail = w == 0ull || (minp && !minp_pass(z, m_t, P.log_min_p));
          const float zs = __fsub_rn(z, score_top);
          if (!fail && zs > -kGumbelMax) {
            const float tt = fminf(expf(zs) * (1.0f + 1.0f / 128.0f), 1.0f) * 33554432.0f;
            const uint32_t T = (uint32_t)ceilf(tt);
            bmin = T >= 33554431u ? 0u : ((33554431u - T) >> 1) + 1u;
          }
        }
        if (fail) {
          dm = min(dm, d);
          w = 0ull;
        }
      }
      wt[d] = w;
      bt[d] = bmin;
    }
    atomicMin(&s.dmin, dm);
  }
  __syncthreads();
  if (tid == 0) {
    R.tau_x = tau_x;
    R.tau16 = tau16;
    R.cmax = cmax;
    R.tiny = tiny;
    R.dcut = s.dmin;
    R.score_top = score_top;
    R.lastkey = 0ull;
    R.route = kRouteHist;
  }
}

// ---------------------------------------------------------------------------
// P3: per-slice collection (the second read of the slice, from L2)
// ---------------------------------------------------------------------------
struct CollectSmem {
  unsigned int cnt[kCodeSlots];   // top-p rows: survivors per regular code slot
  uint32_t bthr[kCodeSlots];      // top-p rows: the row's noise-bits thresholds per slot
  uint64_t cand[kSliceCand];
  Contender cont[kSliceCont];
  unsigned long long tiny_mass, catch_mass;
  unsigned int tiny_cnt, catch_cnt;
  int ncand, ncont;
  uint32_t base;
  RedSmem red;
};

// The rare paths of the element loop, out of line (the loop stays small).
__device__ __noinline__ void stage_cands(CollectSmem& s, uint4 v, int j0, float tau_x,
                                         float inv_t) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float xe = val_of(v, e);
    if (xe >= tau_x) {
      const int pos = atomicAdd(&s.ncand, 1);
      if (pos < kSliceCand) s.cand[pos] = elem_key(__fmul_rn(xe, inv_t), (uint32_t)(j0 + e));
    }
  }
}

// An element of the code-0 slot or of the catch-all (several values each):
// exact min-p and mass per element.  Returns whether it survives with mass > 0.
__device__ __noinline__ bool special_slot(CollectSmem& s, bool is_tiny, float z, float m_t,
                                          bool minp, double lmp) {
  const unsigned long long w = (!minp || minp_pass(z, m_t, lmp)) ? mass_fixed(z, m_t) : 0ull;
  if (w == 0ull) return false;
  if (is_tiny) {
    atomicAdd(&s.tiny_cnt, 1u);
    atomicAdd(&s.tiny_mass, w);
  } else {
    atomicAdd(&s.catch_cnt, 1u);
    atomicAdd(&s.catch_mass, w);
  }
  return true;
}

// The exact score of an element the certificate could not rule out; a
// contender when it beats the maximum's score.
__device__ __noinline__ void try_contender(CollectSmem& s, float z, int j, uint32_t b,
                                           float score_top, int argj, int d) {
  const float sc = gumbel_score(z, b);
  if (!pair_better(sc, j, score_top, argj)) return;
  const int pos = atomicAdd(&s.ncont, 1);
  if (pos < kSliceCont) {
    Contender ct;
    ct.score = sc;
    ct.j = j;
    ct.z = z;
    ct.d = d;
    s.cont[pos] = ct;
  }
}

template <int NV>
__global__ void __launch_bounds__(kFT) flat_collect_kernel(const FlatArgs a) {
  __shared__ CollectSmem s;
  const int sl = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
  const FlatMem M = carve(a.scratch, a.B, a.C);
  FlatRow* Rp = M.rows + row;
  const int route = Rp->route;
  if (route != kRouteCand && route != kRouteHist) return;  // uniform over the CTA
  const int lo = sl * a.L, hi = min(a.V, lo + a.L);
  const bool hist = route == kRouteHist;
  // on candidate rows only the threads whose maximum reached tau read again
  const bool mine = hist || M.tmax[((size_t)row * a.C + sl) * kFT + tid] >= Rp->tau16;
  if (!hist && !__syncthreads_or(mine)) return;  // no candidate in this slice
  const int nvec = mine ? (hi - lo + 7) >> 3 : 0;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(a.logits) + (int64_t)row * a.ld;
  uint4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = tid + i * kFT;
    v[i] = c < nvec ? load_vec(x, lo, hi, c) : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
  const FlatRow R = *Rp;
  const RowParams P = a.params[row];
  const bool topp = hist && (P.flags & kRowTopP) != 0;
  const bool minp = (P.flags & kRowMinP) != 0;
  if (topp) {
    const uint32_t* bt = M.btab + (size_t)row * kCodeSlots;
    for (int d = tid; d < kCodeSlots; d += kFT) {
      s.cnt[d] = 0u;
      s.bthr[d] = bt[d];
    }
  }
  if (tid == 0) {
    s.ncand = 0;
    s.ncont = 0;
    s.tiny_mass = s.catch_mass = 0ull;
    s.tiny_cnt = s.catch_cnt = 0u;
  }
  __syncthreads();
  const float inv_t = P.inv_t, m_t = R.m_t, tau_x = R.tau_x, score_top = R.score_top;
  const double lmp = P.log_min_p;
  const int cmax = R.cmax, tiny = R.tiny, dcut = R.dcut, argj = R.argj;
  const uint64_t key = hist ? row_key(a.seeds[row], row) : 0ull;
  // an element whose z_t is below this cannot out-score the maximum
  const float zfloor = __fsub_rn(score_top, kGumbelMax);
  uint32_t surv = 0u;
  unsigned long long lastk = 0ull;  // max of ~key over survivors
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint4 cur = v[i];
    const int c = tid + i * kFT;
    if (c >= nvec) break;
    const int j0 = lo + 8 * c;
    const float vm = vec_max(cur);
    if (vm >= tau_x) stage_cands(s, cur, j0, tau_x, inv_t);
    if (!hist || !(vm > -INFINITY)) continue;
    // counter of the vector's first column pair; the next pairs add the step
    const uint64_t hbase = key + kSeedStep * ((uint64_t)(j0 >> 1) + 1ull);
    // one column pair (one 32-bit word of the vector) an iteration: the loop
    // body is emitted once per vector
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const uint32_t w = q < 2 ? (q == 0 ? cur.x : cur.y) : (q == 2 ? cur.z : cur.w);
      const uint32_t uh[2] = {w & 0xFFFFu, w >> 16};
      const int je = j0 + 2 * q;
      if (topp) {
        // per element: its slot, the count, and the bits from which it may
        // out-score the maximum (2^24: never; special slots decide exactly)
        uint32_t bneed[2];
        int d[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t u = uh[h];
          bneed[h] = 1u << 24;
          d[h] = 0;
          if (u == 0xFF80u) continue;  // -inf
          const int dd = cmax - code16(u);
          if (dd < dcut && dd != tiny) {
            atomicAdd(&s.cnt[dd], 1u);
            bneed[h] = s.bthr[dd];
            d[h] = dd;
          } else if (dd == tiny || dd >= kCodeSlots - 1) {
            const float ze = __fmul_rn(__uint_as_float(u << 16), inv_t);
            if (special_slot(s, dd == tiny, ze, m_t, minp, lmp)) bneed[h] = 0u;
            d[h] = dd >= kCodeSlots - 1 ? kCodeSlots - 1 : dd;
          }
        }
        if (bneed[0] < (1u << 24) || bneed[1] < (1u << 24)) {
          const uint64_t hsh = sm64_mix(hbase + kSeedStep * (uint64_t)q);
          const uint32_t b0 = bits_even(hsh), b1 = bits_odd(hsh);
          if (b0 >= bneed[0])
            try_contender(s, __fmul_rn(__uint_as_float(uh[0] << 16), inv_t), je, b0, score_top,
                          argj, d[0]);
          if (b1 >= bneed[1])
            try_contender(s, __fmul_rn(__uint_as_float(uh[1] << 16), inv_t), je + 1, b1,
                          score_top, argj, d[1]);
        }
        continue;
      }
      bool sv[2];
      float z[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float xe = __uint_as_float(uh[h] << 16);
        z[h] = __fmul_rn(xe, inv_t);
        sv[h] = xe > -INFINITY && (!minp || minp_pass(z[h], m_t, lmp));
        if (sv[h]) {
          ++surv;
          const unsigned long long nk = ~elem_key(z[h], (uint32_t)(je + h));
          lastk = nk > lastk ? nk : lastk;
        }
      }
      // contenders: survivors whose score beats the maximum's
      const bool t0 = sv[0] && z[0] >= zfloor, t1 = sv[1] && z[1] >= zfloor;
      if (t0 || t1) {
        const uint64_t hsh = sm64_mix(hbase + kSeedStep * (uint64_t)q);
        if (t0 && may_beat(z[0], score_top, bits_even(hsh)))
          try_contender(s, z[0], je, bits_even(hsh), score_top, argj, 0);
        if (t1 && may_beat(z[1], score_top, bits_odd(hsh)))
          try_contender(s, z[1], je + 1, bits_odd(hsh), score_top, argj, 0);
      }
    }
  }
  __syncthreads();
  // flush the staged candidates and contenders to the row's lists
  const int nc = s.ncand, nt = s.ncont;
  if (tid == 0) {
    uint32_t ovf = (nc > kSliceCand || nt > kSliceCont) ? 1u : 0u;
    s.base = 0u;
    if (!ovf && nc > 0) {
      s.base = atomicAdd(&Rp->ncand, (uint32_t)nc);
      if (s.base + (uint32_t)nc > (uint32_t)kFlatCandCap) ovf = 1u;
    }
    if (ovf) atomicOr(&Rp->overflow, 1u);
  }
  __syncthreads();
  if (nc <= kSliceCand && s.base + (uint32_t)nc <= (uint32_t)kFlatCandCap) {
    uint64_t* dst = M.cand + (size_t)row * kFlatCandCap + s.base;
    for (int i = tid; i < nc; i += kFT) dst[i] = s.cand[i];
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t ovf = nt > kSliceCont ? 1u : 0u;
    s.base = 0u;
    if (nt > 0 && nt <= kSliceCont) {
      s.base = atomicAdd(&Rp->ncont, (uint32_t)nt);
      if (s.base + (uint32_t)nt > (uint32_t)kFlatContCap) ovf = 1u;
    }
    if (ovf) atomicOr(&Rp->overflow, 1u);
  }
  __syncthreads();
  if (nt <= kSliceCont && s.base + (uint32_t)nt <= (uint32_t)kFlatContCap) {
    Contender* dst = M.cont + (size_t)row * kFlatContCap + s.base;
    for (int i = tid; i < nt; i += kFT) dst[i] = s.cont[i];
  }
  if (!hist) return;  // uniform
  if (!topp) {
    const unsigned long long sv_all = bsum_u64<kFT>((unsigned long long)surv, s.red);
    const unsigned long long lk = bmax_u64<kFT>(lastk, s.red);
    if (tid == 0) {
      if (sv_all) atomicAdd(&Rp->surv, (uint32_t)sv_all);
      if (lk) atomicMax(&Rp->lastkey, lk);
    }
    return;
  }
  // top-p rows: 64 coarse bins of 64 slots, exact fixed-point masses
  __syncthreads();
  unsigned long long bm = 0ull;
  uint32_t bc = 0u;
  const int d0 = tid * (kCodeSlots / kFT);
#pragma unroll 1
  for (int q = 0; q < kCodeSlots / kFT; ++q) {
    const int d = d0 + q;
    if (d == tiny) {
      bm += s.tiny_mass;
      bc += s.tiny_cnt;
    } else if (d == kCodeSlots - 1) {
      bm += s.catch_mass;
      bc += s.catch_cnt;
    } else {
      const unsigned int k = s.cnt[d];
      if (k) {
        bm += (unsigned long long)k * M.wtab[(size_t)row * kCodeSlots + d];
        bc += k;
      }
    }
  }
  // 4 threads a bin
  bm += __shfl_xor_sync(0xffffffffu, bm, 1);
  bc += __shfl_xor_sync(0xffffffffu, bc, 1);
  bm += __shfl_xor_sync(0xffffffffu, bm, 2);
  bc += __shfl_xor_sync(0xffffffffu, bc, 2);
  FlatHist* H = M.hist + (size_t)row * a.C + sl;
  if ((tid & 3) == 0) {
    H->mass[tid >> 2] = bm;
    H->cnt[tid >> 2] = bc;
  }
  if (tid == 0) {
    H->tiny_mass = s.tiny_mass;
    H->catch_mass = s.catch_mass;
    H->tiny_cnt = s.tiny_cnt;
    H->catch_cnt = s.catch_cnt;
  }
}

// ---------------------------------------------------------------------------
// P4: per-row completion on the candidates (and the top-p boundary bin)
// ---------------------------------------------------------------------------
struct FinishSmem {
  uint64_t keys[kFlatCandCap];     // the row's candidates, unsorted
  uint64_t sel[kFlatKMax];         // a selected prefix, sorted
  unsigned long long bmass[kFlatBins];
  uint32_t bcnt[kFlatBins];
  unsigned int hist[256];
  int bin, rank, nsel;
  uint64_t found;
  RedSmem red;
};

// The r-th largest of the distinct keys keys[0, n) (1 <= r <= n): a
// most-significant-byte radix selection, stopping once one key is left.
__device__ uint64_t select_desc(const uint64_t* keys, int n, int r, FinishSmem& s) {
  uint64_t prefix = 0ull, mask = 0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += kF4) s.hist[b] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kF4) {
      const uint64_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&s.hist[(k >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bin_desc(s.hist, r, &s.bin, &s.rank);
    __syncthreads();
    const int b = max(s.bin, 0);  // (r never exceeds the keys matching the prefix)
    const unsigned int in_bin = s.hist[b];
    prefix |= (uint64_t)b << shift;
    mask |= 0xFFull << shift;
    r = s.rank;
    if (in_bin == 1u) {
      for (int i = threadIdx.x; i < n; i += kF4)
        if ((keys[i] & mask) == prefix) s.found = keys[i];
      __syncthreads();
      return s.found;
    }
    __syncthreads();
  }
  return prefix;
}

// Copy the keys >= kmin (exactly m of them) into s.sel and sort them
// descending (m <= kFlatKMax).
__device__ void gather_sorted(const uint64_t* keys, int n, uint64_t kmin, int m, FinishSmem& s) {
  int P2 = 64;
  while (P2 < m) P2 <<= 1;
  if (threadIdx.x == 0) s.nsel = 0;
  for (int i = threadIdx.x; i < P2; i += kF4) s.sel[i] = 0ull;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kF4) {
    const uint64_t k = keys[i];
    if (k >= kmin) s.sel[atomicAdd(&s.nsel, 1)] = k;
  }
  __syncthreads();
  smem_sort_desc<kF4>(s.sel, P2);
}

__global__ void __launch_bounds__(kF4) flat_finish_kernel(const FlatArgs a) {
  __shared__ FinishSmem s;
  const int row = blockIdx.x, tid = threadIdx.x;
  const FlatMem M = carve(a.scratch, a.B, a.C);
  FlatRow* Rp = M.rows + row;
  const FlatRow R = *Rp;
  if (R.route != kRouteCand && R.route != kRouteHist) return;
  if (R.overflow) {
    if (tid == 0) hand_over(a, *Rp, row, false);
    return;
  }
  const RowParams P = a.params[row];
  const int n = a.n_logprobs;
  const float m_t = R.m_t, lnS = R.lnS;
  const int nc = (int)min(R.ncand, (uint32_t)kFlatCandCap);
  const uint64_t* src = M.cand + (size_t)row * kFlatCandCap;
  // few candidates are sorted outright; more are selected from
  const bool small = nc <= kSmallCand;
  {
    int P2 = small ? 64 : nc;
    while (small && P2 < nc) P2 <<= 1;
    for (int i = tid; i < P2; i += kF4) s.keys[i] = i < nc ? src[i] : 0ull;
    __syncthreads();
    if (small && nc > 1) smem_sort_desc<kF4>(s.keys, P2);
  }
  // top-n: the candidates hold the row's n largest
  if (n > 0) {
    const uint64_t* top = s.keys;
    if (!small) {
      const uint64_t kn = select_desc(s.keys, nc, n, s);
      gather_sorted(s.keys, nc, kn, n, s);
      top = s.sel;
    }
    for (int t = tid; t < n; t += kF4) {
      const uint64_t k = top[t];
      a.out_topk_ids[(int64_t)row * n + t] = (int)key_idx(k);
      a.out_topk_logprobs[(int64_t)row * n + t] = (key_z(k) - m_t) - lnS;
    }
    __syncthreads();
  }
  const bool greedy = (P.flags & kRowGreedy) != 0;
  if (R.route == kRouteCand) {
    if (greedy) {
      if (tid == 0) {
        write_row(a, row, R.argj, m_t, m_t, lnS, m_t, R.argj, 1);
        Rp->route = kRouteDone;
      }
      return;
    }
    // min-p, then top-k, then top-p over the top-k survivors renormalised:
    // the candidates hold at least top_k elements and are a prefix of the
    // row's order, so each cut falls inside them
    int L1 = nc;
    if (P.flags & kRowMinP) {
      int pass = 0;
      for (int i = tid; i < nc; i += kF4) pass += minp_pass(key_z(s.keys[i]), m_t, P.log_min_p);
      L1 = (int)bsum_u64<kF4>((unsigned long long)pass, s.red);
    }
    const int L2 = min(P.top_k, L1);
    const bool topp = (P.flags & kRowTopP) != 0;
    // the kept prefix in order: the sorted candidates, or the L2 largest
    // selected and sorted (only top-p needs their order)
    const uint64_t* ord = s.keys;
    uint64_t k2;
    if (small) {
      k2 = s.keys[L2 - 1];
    } else {
      k2 = select_desc(s.keys, nc, L2, s);
      if (topp) {
        gather_sorted(s.keys, nc, k2, L2, s);
        ord = s.sel;
      }
    }
    int L3 = L2;
    uint64_t kth = k2;
    if (topp) {
      const int per = (L2 + kF4 - 1) / kF4;
      const int i0 = min(L2, tid * per), i1 = min(L2, i0 + per);
      unsigned long long mine = 0ull;
      for (int i = i0; i < i1; ++i) mine += mass_fixed(key_z(ord[i]), m_t);
      unsigned long long W = 0ull;
      unsigned long long run = bexscan_u64<kF4>(mine, &W, s.red);
      const unsigned long long Tm = (unsigned long long)((double)W * (double)P.top_p);
      int kept = 0;
      for (int i = i0; i < i1; ++i) {
        if (run <= Tm) ++kept;
        run += mass_fixed(key_z(ord[i]), m_t);
      }
      L3 = max(1, (int)bsum_u64<kF4>((unsigned long long)kept, s.red));
      kth = ord[L3 - 1];
    }
    // the Gumbel-max draw over the kept set: the first L3 in order (top-p or
    // sorted), else the candidates at or above the L2-th
    const uint64_t key = row_key(a.seeds[row], row);
    float bs = -INFINITY, bz = 0.f;
    int bj = INT_MAX;
    const bool prefix = topp || small;
    const int span = prefix ? L3 : nc;
    for (int i = tid; i < span; i += kF4) {
      const uint64_t k = ord[i];
      if (!prefix && k < k2) continue;
      const int j = (int)key_idx(k);
      const float z = key_z(k);
      const float sc = gumbel_score_inl(z, noise_bits(key, j));
      if (pair_better(sc, j, bs, bj)) {
        bs = sc;
        bj = j;
        bz = z;
      }
    }
    bargmax<kF4>(bs, bj, bz, s.red);
    if (tid == 0) {
      write_row(a, row, bj, bz, m_t, lnS, key_z(kth), (int)key_idx(kth), L3);
      Rp->route = kRouteDone;
    }
    return;
  }
  // rows without top-k
  if (!(P.flags & kRowTopP)) {
    // kept: every survivor; the winner: the best contender, else the maximum
    const int nt = (int)min(R.ncont, (uint32_t)kFlatContCap);
    const Contender* ct = M.cont + (size_t)row * kFlatContCap;
    float bs = -INFINITY, bz = 0.f;
    int bj = INT_MAX;
    for (int i = tid; i < nt; i += kF4) {
      const Contender c = ct[i];
      if (pair_better(c.score, c.j, bs, bj)) {
        bs = c.score;
        bj = c.j;
        bz = c.z;
      }
    }
    bargmax<kF4>(bs, bj, bz, s.red);
    if (tid == 0) {
      const int tok = bj == INT_MAX ? R.argj : bj;
      const float ztok = bj == INT_MAX ? m_t : bz;
      const uint64_t last = ~R.lastkey;
      write_row(a, row, tok, ztok, m_t, lnS, key_z(last), (int)key_idx(last), (int)R.surv);
      Rp->route = kRouteDone;
    }
    return;
  }
  // top-p rows: the coarse bin where the prefix mass first exceeds floor(W p)
  {
    const int b = tid >> 2, part = tid & 3;  // 4 threads a bin
    unsigned long long m = 0ull;
    uint32_t c = 0u;
    for (int sl = part; sl < a.C; sl += 4) {
      const FlatHist* H = M.hist + (size_t)row * a.C + sl;
      m += H->mass[b];
      c += H->cnt[b];
    }
    m += __shfl_xor_sync(0xffffffffu, m, 1);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    m += __shfl_xor_sync(0xffffffffu, m, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    if (part == 0) {
      s.bmass[b] = m;
      s.bcnt[b] = c;
    }
  }
  __syncthreads();
  if (tid < 32) {
    // lane l owns bins 2l, 2l + 1
    const unsigned long long m0 = s.bmass[2 * tid], m1 = s.bmass[2 * tid + 1];
    const uint32_t c0 = s.bcnt[2 * tid], c1 = s.bcnt[2 * tid + 1];
    unsigned long long inc = m0 + m1;
    uint32_t cinc = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
      const uint32_t ct = __shfl_up_sync(0xffffffffu, cinc, o);
      if (tid >= o) {
        inc += t;
        cinc += ct;
      }
    }
    const unsigned long long W = __shfl_sync(0xffffffffu, inc, 31);
    const unsigned long long Tm = (unsigned long long)((double)W * (double)P.top_p);
    const unsigned long long ex = inc - (m0 + m1);
    const uint32_t cex = cinc - (c0 + c1);
    // the first bin whose inclusive prefix exceeds Tm
    const bool in0 = ex + m0 > Tm, in1 = !in0 && ex + m0 + m1 > Tm;
    const unsigned hit = __ballot_sync(0xffffffffu, in0 || in1);
    const int owner = hit ? __ffs(hit) - 1 : 31;
    if (tid == owner) {
      const bool first = hit ? in0 : false;
      Rp->bstar = first ? 2 * tid : 2 * tid + 1;
      Rp->above = first ? ex : ex + m0;
      Rp->cabove = first ? cex : cex + c0;
      Rp->tm = Tm;
      Rp->route = kRouteFine;
    }
  }
}

// ---------------------------------------------------------------------------
// P5: top-p rows, counts per code slot of the boundary bin (a third read)
// ---------------------------------------------------------------------------
template <int NV>
__global__ void __launch_bounds__(kFT) flat_fine_kernel(const FlatArgs a) {
  __shared__ unsigned int cnt[kFlatBins];
  const int sl = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
  const FlatMem M = carve(a.scratch, a.B, a.C);
  const FlatRow* Rp = M.rows + row;
  if (Rp->route != kRouteFine) return;
  const int lo = sl * a.L, hi = min(a.V, lo + a.L);
  const int nvec = (hi - lo + 7) >> 3;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(a.logits) + (int64_t)row * a.ld;
  uint4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = tid + i * kFT;
    v[i] = c < nvec ? load_vec(x, lo, hi, c) : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
  if (tid < kFlatBins) cnt[tid] = 0u;
  __syncthreads();
  const int d0 = Rp->bstar * kFlatBins, cmax = Rp->cmax, tiny = Rp->tiny, dcut = Rp->dcut;
  // codes of the bin's regular survivor slots: (cmax - d0 - 63, cmax - d0]
  const int chi = cmax - d0, clo = cmax - min(d0 + kFlatBins, min(dcut, kCodeSlots - 1)) + 1;
  // the bin's values lie in [code_value(clo), code_value(chi)] (clo <= chi,
  // neither the code-0 slot when the range holds it)
  const float xhi = chi == 0 ? 0.f : code_value(chi), xlo = clo == 0 ? 0.f : code_value(clo);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float xe = val_of(v[i], e);
      if (xe >= xlo && xe <= xhi) {
        const int code = code16(bits_of(v[i], e));
        if (code <= chi && code >= clo && cmax - code != tiny) atomicAdd(&cnt[chi - code], 1u);
      }
    }
  }
  __syncthreads();
  if (tid < kFlatBins) M.fine[((size_t)row * a.C + sl) * kFlatBins + tid] = cnt[tid];
}

// ---------------------------------------------------------------------------
// P6: top-p rows, the boundary slot, the boundary element and the draw
// ---------------------------------------------------------------------------
struct TopPSmem {
  unsigned long long mq[kFlatBins];
  uint32_t cq[kFlatBins];
  uint32_t fslot[kFlatMaxC];   // the boundary slot's count per slice
  RedSmem red;
  int qstar, sstar, tprime, jb, hand;
  uint32_t kept;
  int wcount[kFW];
};

template <int NV>
__global__ void __launch_bounds__(kFT) flat_topp_kernel(const FlatArgs a) {
  __shared__ TopPSmem s;
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const FlatMem M = carve(a.scratch, a.B, a.C);
  FlatRow* Rp = M.rows + row;
  const FlatRow R = *Rp;
  if (R.route != kRouteFine) return;
  const RowParams P = a.params[row];
  const float m_t = R.m_t, lnS = R.lnS, inv_t = P.inv_t;
  const int d0 = R.bstar * kFlatBins, cmax = R.cmax, tiny = R.tiny, dcut = R.dcut;
  // per slot of the bin: survivors and their mass (the counts of the C slices
  // summed by 4 threads a slot)
  {
    const int q = tid >> 2, part = tid & 3;
    const int d = d0 + q;
    unsigned long long mq = 0ull;
    uint32_t cq = 0u;
    if (d == tiny || d == kCodeSlots - 1) {
      for (int sl = part; sl < a.C; sl += 4) {
        const FlatHist* H = M.hist + (size_t)row * a.C + sl;
        mq += d == tiny ? H->tiny_mass : H->catch_mass;
        cq += d == tiny ? H->tiny_cnt : H->catch_cnt;
      }
    } else if (d < dcut) {
      for (int sl = part; sl < a.C; sl += 4) cq += M.fine[((size_t)row * a.C + sl) * kFlatBins + q];
    }
    mq += __shfl_xor_sync(0xffffffffu, mq, 1);
    cq += __shfl_xor_sync(0xffffffffu, cq, 1);
    mq += __shfl_xor_sync(0xffffffffu, mq, 2);
    cq += __shfl_xor_sync(0xffffffffu, cq, 2);
    if (part == 0) {
      if (d != tiny && d != kCodeSlots - 1 && cq)
        mq = (unsigned long long)cq * M.wtab[(size_t)row * kCodeSlots + d];
      s.mq[q] = mq;
      s.cq[q] = cq;
    }
  }
  __syncthreads();
  if (tid < 32) {
    const unsigned long long Tm = R.tm;
    const unsigned long long m0 = s.mq[2 * tid], m1 = s.mq[2 * tid + 1];
    const uint32_t c0 = s.cq[2 * tid], c1 = s.cq[2 * tid + 1];
    unsigned long long inc = m0 + m1;
    uint32_t cinc = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
      const uint32_t ct = __shfl_up_sync(0xffffffffu, cinc, o);
      if (tid >= o) {
        inc += t;
        cinc += ct;
      }
    }
    const unsigned long long ex = R.above + inc - (m0 + m1);
    const uint32_t cex = R.cabove + cinc - (c0 + c1);
    const bool in0 = ex + m0 > Tm, in1 = !in0 && ex + m0 + m1 > Tm;
    const unsigned hit = __ballot_sync(0xffffffffu, in0 || in1);
    const int owner = hit ? __ffs(hit) - 1 : 31;
    if (tid == owner) {
      const bool first = hit ? in0 : false;
      const int q = first ? 2 * tid : 2 * tid + 1;
      const unsigned long long A = first ? ex : ex + m0;
      const uint32_t cA = first ? cex : cex + c0;
      const int d = d0 + q;
      s.qstar = q;
      s.hand = (!hit || d == tiny || d >= kCodeSlots - 1 || s.cq[q] == 0u) ? 1 : 0;
      if (!s.hand) {
        const unsigned long long w = M.wtab[(size_t)row * kCodeSlots + d];
        const unsigned long long t = min((unsigned long long)s.cq[q], (Tm - A) / w + 1ull);
        s.kept = cA + (uint32_t)t;
        s.tprime = (int)t;
      }
      s.jb = INT_MAX;
    }
  }
  __syncthreads();
  if (s.hand) {
    if (tid == 0) hand_over(a, *Rp, row, a.n_logprobs > 0);
    return;
  }
  const int q = s.qstar, dstar = d0 + q;
  const int cstar = cmax - dstar;  // the boundary slot's code
  // the slice holding the tprime-th element of the slot, in index order
  if (tid < a.C) s.fslot[tid] = M.fine[((size_t)row * a.C + tid) * kFlatBins + q];
  __syncthreads();
  if (tid == 0) {
    int left = s.tprime, sl = 0;
    for (; sl < a.C - 1; ++sl) {
      if (left <= (int)s.fslot[sl]) break;
      left -= (int)s.fslot[sl];
    }
    s.sstar = sl;
    s.tprime = left;
  }
  __syncthreads();
  // its tprime-th element of code cstar: the slice's vectors in index order
  // (vector c = thread + i * kFT), one block scan per register vector
  {
    const int lo = s.sstar * a.L, hi = min(a.V, lo + a.L);
    const int nvec = (hi - lo + 7) >> 3;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(a.logits) + (int64_t)row * a.ld;
    uint4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = tid + i * kFT;
      v[i] = c < nvec ? load_vec(x, lo, hi, c) : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
    }
    const int want = s.tprime;
    int seen = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      uint32_t mask = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t u = bits_of(v[i], e);
        if (u != 0xFF80u && code16(u) == cstar) mask |= 1u << e;
      }
      const int m = __popc(mask);
      int inc = m;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (lane == 31) s.wcount[warp] = inc;
      __syncthreads();
      int before = seen, total = 0;
#pragma unroll
      for (int w = 0; w < kFW; ++w) {
        if (w < warp) before += s.wcount[w];
        total += s.wcount[w];
      }
      before += inc - m;
      if (m > 0 && before < want && want <= before + m) {
        int r = want - before;  // 1-based within this vector
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if ((mask >> e) & 1u) {
            if (--r == 0) s.jb = lo + 8 * (tid + i * kFT) + e;
          }
        }
      }
      seen += total;
      __syncthreads();
    }
  }
  const int jb = s.jb;
  if (jb == INT_MAX) {  // counts and scan disagree: leave the row to the selection kernel
    if (tid == 0) hand_over(a, *Rp, row, a.n_logprobs > 0);
    return;
  }
  // the winner: the best kept contender, else the maximum
  const int nt = (int)min(R.ncont, (uint32_t)kFlatContCap);
  const Contender* ct = M.cont + (size_t)row * kFlatContCap;
  float bs = -INFINITY, bz = 0.f;
  int bj = INT_MAX;
  for (int i = tid; i < nt; i += kFT) {
    const Contender c = ct[i];
    const bool kept = c.d < dstar || (c.d == dstar && c.j <= jb);
    if (kept && pair_better(c.score, c.j, bs, bj)) {
      bs = c.score;
      bj = c.j;
      bz = c.z;
    }
  }
  bargmax<kFT>(bs, bj, bz, s.red);
  if (tid == 0) {
    const int tok = bj == INT_MAX ? R.argj : bj;
    const float ztok = bj == INT_MAX ? m_t : bz;
    write_row(a, row, tok, ztok, m_t, lnS, __fmul_rn(code_value(cstar), inv_t), jb,
              (int)s.kept);
    Rp->route = kRouteDone;
  }
}

template <int NV>
cudaError_t launch_nv(const FlatArgs& a, cudaStream_t stream) {
  const dim3 grid((unsigned)a.C, (unsigned)a.B);
  flat_stats_kernel<NV><<<grid, kFT, 0, stream>>>(a);
  flat_row_kernel<<<a.B, kFF, 0, stream>>>(a);
  flat_collect_kernel<NV><<<grid, kFT, 0, stream>>>(a);
  flat_finish_kernel<<<a.B, kF4, 0, stream>>>(a);
  flat_fine_kernel<NV><<<grid, kFT, 0, stream>>>(a);
  flat_topp_kernel<NV><<<a.B, kFT, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

// Slices of at most kFlatSlice elements (the slice's vectors stay in
// registers), at most kFlatMaxC per row.
FlatPlan plan_flat(int V) {
  FlatPlan p{0, 0, 0};
  if (V < 1) return p;
  int C = (V + kFlatSlice - 1) / kFlatSlice;
  if (C > kFlatMaxC) C = kFlatMaxC;
  int L = (V + C - 1) / C;
  L = (L + 7) & ~7;
  const int NV = ((L / 8) + kFT - 1) / kFT;
  if (NV > kFlatMaxNV) return p;
  p.C = C;
  p.L = L;
  p.NV = NV;
  return p;
}

size_t flat_scratch_bytes(int B, int C) { return carve_bytes(B, C); }

cudaError_t launch_flat(const FlatArgs& a, cudaStream_t stream) {
  if (a.B < 1) return cudaSuccess;
  switch (a.NV) {
    case 1: return launch_nv<1>(a, stream);
    case 2: return launch_nv<2>(a, stream);
    case 3: return launch_nv<3>(a, stream);
    case 4: return launch_nv<4>(a, stream);
    case 5: return launch_nv<5>(a, stream);
    case 6: return launch_nv<6>(a, stream);
    case 7: return launch_nv<7>(a, stream);
    case 8: return launch_nv<8>(a, stream);
    case 9: return launch_nv<9>(a, stream);
    case 10: return launch_nv<10>(a, stream);
    case 11: return launch_nv<11>(a, stream);
    case 12: return launch_nv<12>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vt
