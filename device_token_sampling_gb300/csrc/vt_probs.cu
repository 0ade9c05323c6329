// vt_probs.cu -- the filtered distribution a sampling call drew from, on
// request [TensorRT-LLM "Sampling", Performance: the complete set of token
// probabilities after the top-k / top-p masking is skipped by the sorting-free
// path unless the user asks for it, e.g. for rejection sampling].
//
// For a row the call sampled, p_j = exp(z_t,j - m) / sum_kept exp(z_t - m) for
// j in the kept set (the prefix of the order (z_t descending, index
// ascending) that ends at the boundary element the call recorded), 0
// elsewhere; m is the row maximum, which the kept set always holds.  A greedy
// row gets a one-hot vector at its token, a row the call could not sample
// (status != 0) gets NaN everywhere.
//
// Two launches over (row, split) CTAs, each split a contiguous range of the
// row: the first streams its range once for the kept elements' maximum and
// their exp-sum relative to it (online rescaling), the second combines the
// row's partials and streams the range again to write fp32 probabilities.
// Both recompute z_t with the sampling kernels' arithmetic (the penalised
// value of a seen id, times 1/T, each rounded once), so that the kept test
// against the recorded boundary is exact.  The work is HBM-bound: per row it
// reads the logits twice and writes 4 bytes per entry.
#include <cstdint>

#include "vt_device.cuh"
#include "vt_kernels.h"

namespace vt {
namespace {

constexpr int kPThreads = 256;
constexpr int kUnroll = 4;  // 16-byte loads in flight per thread

template <typename T>
struct Vec;

template <>
struct Vec<float> {
  static constexpr int E = 4;
  __device__ static void load(const float* p, float* x) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    x[0] = __uint_as_float(a.x);
    x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z);
    x[3] = __uint_as_float(a.w);
  }
  __device__ static float load1(const float* p) { return __ldg(p); }
};

// bfloat16 as its 16 bits: widening to fp32 is exact.
template <>
struct Vec<uint16_t> {
  static constexpr int E = 8;
  __device__ static void load(const uint16_t* p, float* x) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static float load1(const uint16_t* p) {
    return __uint_as_float((uint32_t)__ldg(p) << 16);
  }
};

// First entry of the sorted (id, count) table whose id is >= id.
__device__ __forceinline__ int lower_bound_id(const int2* tab, int len, int id) {
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid].x < id) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// (max, sum) pairs: the sum is relative to the max; (-inf, 0) is empty.
__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s = s + s2 * expf(m2 - m);
  }
}

struct RowSetup {
  int lo, hi;          // this CTA's range of the row
  int e_lo, e_hi;      // its seen ids in the count table
  const int2* tab;
};

// The CTA's range and its slice of the count table (rows with penalties).
__device__ __forceinline__ RowSetup row_setup(const ProbsArgs& a, int row, int split,
                                              const RowParams& P, int* sh) {
  RowSetup r;
  r.lo = split * a.range;
  r.hi = min(r.lo + a.range, a.V);
  r.tab = a.hist + (int64_t)row * a.hist_cap;
  r.e_lo = r.e_hi = 0;
  if ((P.flags & kRowPenalty) && a.hist) {
    if (threadIdx.x == 0) {
      const int len = a.hist_len[row];
      sh[0] = lower_bound_id(r.tab, len, r.lo);
      sh[1] = lower_bound_id(r.tab, len, r.hi);
    }
    __syncthreads();
    r.e_lo = sh[0];
    r.e_hi = sh[1];
  }
  return r;
}

// Visit every element of [lo, hi) as (value, index, vector slot): 16-byte
// loads over the whole vectors (kUnroll in flight per thread), then the tail.
// fn(x[E], j0, n) gets a vector of n <= E values starting at index j0.
template <typename T, typename FN>
__device__ __forceinline__ void stream_range(const T* x, int lo, int hi, bool vec, FN fn) {
  constexpr int E = Vec<T>::E;
  const int nvec = vec ? (hi - lo) / E : 0;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kPThreads * kUnroll) {
    float xs[kUnroll][E];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * kPThreads;
      if (v < nvec) Vec<T>::load(x + lo + v * E, xs[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * kPThreads;
      if (v < nvec) fn(xs[u], lo + v * E, E);
    }
  }
  for (int j = lo + nvec * E + threadIdx.x; j < hi; j += kPThreads) {
    float one[E];
    one[0] = Vec<T>::load1(x + j);
    fn(one, j, 1);
  }
}

template <typename T>
__global__ void __launch_bounds__(kPThreads) probs_stats_kernel(const ProbsArgs a) {
  __shared__ uint32_t bitmap[kProbsMaxRange / 32];
  __shared__ float red_m[kPThreads / 32], red_s[kPThreads / 32];
  __shared__ int sh[2];
  const int row = (int)(blockIdx.x / (unsigned)a.splits);
  const int split = (int)(blockIdx.x % (unsigned)a.splits);
  const RowParams P = a.params[row];
  if (a.row_status[row] != kRowOk || (P.flags & kRowGreedy)) return;  // no partial needed
  const RowSetup rs = row_setup(a, row, split, P, sh);
  const bool pen = rs.e_hi > rs.e_lo;
  if (pen) {  // the range's seen ids, whose values the table entries give
    const int nwords = (rs.hi - rs.lo + 31) >> 5;
    for (int w = threadIdx.x; w < nwords; w += kPThreads) bitmap[w] = 0u;
    __syncthreads();
    for (int e = rs.e_lo + (int)threadIdx.x; e < rs.e_hi; e += kPThreads) {
      const int local = rs.tab[e].x - rs.lo;
      atomicOr(&bitmap[local >> 5], 1u << (local & 31));
    }
    __syncthreads();
  }
  const uint64_t kkey = elem_key(a.kth_value[row], (uint32_t)a.kth_index[row]);
  const float inv_t = P.inv_t;
  float m = -INFINITY, s = 0.0f;
  auto add = [&](float zt, int j) {
    if (zt == -INFINITY || elem_key(zt, (uint32_t)j) < kkey) return;
    if (zt > m) {
      s = s * expf(m - zt) + 1.0f;
      m = zt;
    } else {
      s += expf(zt - m);
    }
  };
  const T* x = reinterpret_cast<const T*>(a.logits) + (int64_t)row * a.ld;
  constexpr int E = Vec<T>::E;
  stream_range<T>(x, rs.lo, rs.hi, a.vec_in != 0, [&](const float* v, int j0, int n) {
    uint32_t skip = 0u;
    if (pen) {
      const int local = j0 - rs.lo;  // E divides 32 and j0 - lo: one word holds the vector
      skip = bitmap[local >> 5] >> (local & 31);
    }
#pragma unroll
    for (int i = 0; i < E; ++i)
      if (i < n && !((skip >> i) & 1u)) add(__fmul_rn(v[i], inv_t), j0 + i);
  });
  for (int e = rs.e_lo + (int)threadIdx.x; e < rs.e_hi; e += kPThreads) {
    const int2 t = rs.tab[e];
    add(__fmul_rn(penalize(Vec<T>::load1(x + t.x), t.y, P), inv_t), t.x);
  }
  // block combine
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    combine(m, s, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY, S = 0.0f;
    for (int w = 0; w < kPThreads / 32; ++w) combine(M, S, red_m[w], red_s[w]);
    a.part[blockIdx.x] = make_float2(M, S);
  }
}

template <typename T>
__global__ void __launch_bounds__(kPThreads) probs_write_kernel(const ProbsArgs a) {
  __shared__ float sMS[2];
  __shared__ int sh[2];
  const int row = (int)(blockIdx.x / (unsigned)a.splits);
  const int split = (int)(blockIdx.x % (unsigned)a.splits);
  const RowParams P = a.params[row];
  float* out = a.probs + (int64_t)row * a.ld_probs;
  const int lo = split * a.range, hi = min(lo + a.range, a.V);
  const int status = a.row_status[row];
  if (status != kRowOk || (P.flags & kRowGreedy)) {  // NaN, or one-hot at the token
    const float fill = status != kRowOk ? __int_as_float(0x7fc00000) : 0.0f;
    const int tok = status != kRowOk ? -1 : a.tokens[row];
    for (int j = lo + (int)threadIdx.x; j < hi; j += kPThreads) out[j] = j == tok ? 1.0f : fill;
    return;
  }
  const RowSetup rs = row_setup(a, row, split, P, sh);
  if (threadIdx.x < 32) {  // the row's (max, sum) from its partials
    float M = -INFINITY, S = 0.0f;
    for (int i = threadIdx.x; i < a.splits; i += 32) {
      const float2 q = a.part[(int64_t)row * a.splits + i];
      combine(M, S, q.x, q.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, M, o);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, S, o);
      combine(M, S, m2, s2);
    }
    if (threadIdx.x == 0) {
      sMS[0] = M;
      sMS[1] = S;
    }
  }
  __syncthreads();
  const float M = sMS[0], S = sMS[1];
  const uint64_t kkey = elem_key(a.kth_value[row], (uint32_t)a.kth_index[row]);
  const float inv_t = P.inv_t;
  auto prob = [&](float zt, int j) {
    if (zt == -INFINITY || elem_key(zt, (uint32_t)j) < kkey) return 0.0f;
    return __fdiv_rn(expf(__fsub_rn(zt, M)), S);
  };
  const T* x = reinterpret_cast<const T*>(a.logits) + (int64_t)row * a.ld;
  constexpr int E = Vec<T>::E;
  const bool vec_out = a.vec_out != 0;
  stream_range<T>(x, lo, hi, a.vec_in != 0, [&](const float* v, int j0, int n) {
    float p[E];
#pragma unroll
    for (int i = 0; i < E; ++i) p[i] = prob(__fmul_rn(v[i], inv_t), j0 + i);
    if (n == E && vec_out) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q)
        reinterpret_cast<float4*>(out + j0)[q] = make_float4(p[4 * q], p[4 * q + 1],
                                                             p[4 * q + 2], p[4 * q + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i)
        if (i < n) out[j0 + i] = p[i];
    }
  });
  if (rs.e_hi > rs.e_lo) {  // the seen ids again, with their penalised values
    __syncthreads();
    for (int e = rs.e_lo + (int)threadIdx.x; e < rs.e_hi; e += kPThreads) {
      const int2 t = rs.tab[e];
      out[t.x] = prob(__fmul_rn(penalize(Vec<T>::load1(x + t.x), t.y, P), inv_t), t.x);
    }
  }
}

}  // namespace

void plan_probs(int B, int V, int num_sms, int* splits, int* range) {
  const int target = kProbsCtasPerSm * num_sms;
  int sp = (target + B - 1) / B;
  const int need = (V + kProbsMaxRange - 1) / kProbsMaxRange;
  if (sp > kProbsMaxSplits) sp = kProbsMaxSplits;
  if (sp < need) sp = need;
  int rg = (V + sp - 1) / sp;
  rg = (rg + 63) / 64 * 64;  // lo stays 16-byte aligned for both element sizes
  if (rg > kProbsMaxRange) rg = kProbsMaxRange;
  *range = rg;
  *splits = (V + rg - 1) / rg;
}

cudaError_t launch_probs(const ProbsArgs& a, int dtype, cudaStream_t st) {
  const unsigned grid = (unsigned)a.B * (unsigned)a.splits;
  if (dtype == 0) {
    probs_stats_kernel<float><<<grid, kPThreads, 0, st>>>(a);
    probs_write_kernel<float><<<grid, kPThreads, 0, st>>>(a);
  } else {
    probs_stats_kernel<uint16_t><<<grid, kPThreads, 0, st>>>(a);
    probs_write_kernel<uint16_t><<<grid, kPThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace vt
