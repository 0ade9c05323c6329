// vt_shard.cu -- the vocabulary-sharded sampler: per-shard partials and their merge.
//
// When the vocabulary of a row is split over several devices (the Tenstorrent
// sampling README: each device takes the top-k of its own slice of the logits,
// the candidates are all-gathered, and the log-probs combine the devices'
// maxima and sums of exponentials -- TTSampling and LogProbsCalculator), the
// draw composes exactly because the noise of column j is keyed by the global
// row and the global column (vllm.cpp pull request: ArgReduce over true global
// indices).  Two launches and one small exchange:
//
//   partials (one per shard): for each row of the shard's columns
//     [v0, v0 + Vs), the shard's tempered maximum m_s, its sum of
//     exp(z_t - m_s), its lowest-index argmax (global index), and its K
//     largest elements as records (z_t, global index) in the order
//     (z_t descending, index ascending);
//   the caller all-gathers the shards' partial buffers (S x B records);
//   merge (any shard, or every shard): the row's maximum and sum of
//     exponentials (hence its log-probs), then min-p, top-k and top-p over the
//     union of the shards' records -- which holds the row's K largest
//     elements -- with masses in exact fixed point, the Gumbel-max draw over
//     the kept records, and the top-n.
//
// The union covers the kept set of every row whose kept set lies inside a
// top-k of at most K (and greedy rows); the host rejects other rows, and any
// S * K above kShardCand (the records one merge CTA sorts).
#include "vt_device.cuh"
#include "vt_kernels.h"
#include "vt_sampler.h"

#include <climits>

namespace vt {
namespace {

constexpr int kST = 256;                 // threads per CTA
constexpr int kSW = kST / 32;
constexpr int kShardCand = 4096;         // records a CTA collects or merges at most

struct __align__(16) ShardHead {
  float m_t;        // the shard's tempered maximum (-inf: no finite element)
  float s;          // sum of exp(z_t - m_t) over the shard
  int32_t argj;     // lowest global index of m_t (INT_MAX: none)
  uint32_t info;    // records written (bits 0..15), NaN or +inf seen (bit 30)
  // rows without a filter (every finite element kept): the shard's Gumbel
  // winner, its finite count and its last finite element in the order
  float wscore;     // the best score z_t - ln(-ln u) (-inf: none)
  int32_t wj;       // its global index (INT_MAX: none)
  float wz;         // its tempered value
  uint32_t nfin;    // finite elements
  unsigned long long last;  // ~key of the last finite element (0: none)
  unsigned long long pad;
};
static_assert(sizeof(ShardHead) == 48, "the documented record header is 48 bytes");

// A row every finite element of which is kept: sampled, without top-k, top-p
// or min-p.
__device__ __forceinline__ bool unfiltered_row(const RowParams& P, int V) {
  const bool greedy = (P.flags & kRowGreedy) != 0;
  const bool topk = P.top_k > 1 && P.top_k < V;
  return !greedy && !topk && !(P.flags & (kRowTopP | kRowMinP));
}

struct ShardSmem {
  uint64_t keys[kShardCand];
  float w_score, w_z;   // merge: the shards' best Gumbel winner (rows without a filter)
  int w_j;
  unsigned int nfin_all;
  unsigned long long last_all;
  uint64_t sel[VT_SHARD_MAX_K];   // the leading records, sorted
  uint64_t found;
  int nsel;
  float tm[kST];
  float rf[2 * kSW];
  int ri[2 * kSW];
  unsigned long long ru[2 * kSW];
  unsigned int hist[256];
  int wt[kSW];
  int count, ties;
  float bf[4];
  int bi[4];
};

// Block argmax (larger value, then lower index).
__device__ void sblock_argmax(float& v, int& i, float& z, ShardSmem& s) {
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
    s.rf[kSW + warp] = z;
  }
  __syncthreads();
  if (warp == 0) {
    float tv = lane < kSW ? s.rf[lane] : -INFINITY;
    int ti = lane < kSW ? s.ri[lane] : INT_MAX;
    float tz = lane < kSW ? s.rf[kSW + lane] : 0.f;
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
      s.bf[0] = tv;
      s.bi[0] = ti;
      s.bf[1] = tz;
    }
  }
  __syncthreads();
  v = s.bf[0];
  i = s.bi[0];
  z = s.bf[1];
  __syncthreads();
}

__device__ float sblock_sum(float v, ShardSmem& s) {
  v = warp_sum_f(v);
  if ((threadIdx.x & 31) == 0) s.rf[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < kSW ? s.rf[threadIdx.x] : 0.f;
    t = warp_sum_f(t);
    if (threadIdx.x == 0) s.bf[2] = t;
  }
  __syncthreads();
  const float r = s.bf[2];
  __syncthreads();
  return r;
}

__device__ unsigned long long sblock_sum_u64(unsigned long long v, ShardSmem& s) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < kSW ? s.ru[threadIdx.x] : 0ull;
    t = warp_sum_u64(t);
    if (threadIdx.x == 0) s.ru[kSW] = t;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kSW];
  __syncthreads();
  return r;
}

__device__ unsigned long long sblock_max_u64(unsigned long long v, ShardSmem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
    v = t > v ? t : v;
  }
  if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long t = threadIdx.x < kSW ? s.ru[threadIdx.x] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long q = __shfl_xor_sync(0xffffffffu, t, o);
      t = q > t ? q : t;
    }
    if (threadIdx.x == 0) s.ru[kSW] = t;
  }
  __syncthreads();
  const unsigned long long r = s.ru[kSW];
  __syncthreads();
  return r;
}

template <typename T>
__device__ __forceinline__ float load_x(const T* p, int j);
template <>
__device__ __forceinline__ float load_x<float>(const float* p, int j) {
  return __ldg(p + j);
}
template <>
__device__ __forceinline__ float load_x<uint16_t>(const uint16_t* p, int j) {
  return __uint_as_float((uint32_t)__ldg(p + j) << 16);
}

// Visit every element j of x[0, n) once, fn(j, value): 16-byte vector loads
// between a scalar head (up to the first 16-byte boundary) and a scalar tail.
// Each thread sees its elements in increasing j.
template <typename T>
__device__ __forceinline__ float vec_elem(const uint4& q, int e);
template <>
__device__ __forceinline__ float vec_elem<float>(const uint4& q, int e) {
  return __uint_as_float(e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w);
}
template <>
__device__ __forceinline__ float vec_elem<uint16_t>(const uint4& q, int e) {
  const uint32_t w = e < 2 ? q.x : e < 4 ? q.y : e < 6 ? q.z : q.w;
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

template <typename T, typename F>
__device__ __forceinline__ void scan_elems(const T* x, int n, F&& fn) {
  constexpr int E = 16 / (int)sizeof(T);
  const int mis = (int)(((uintptr_t)x / sizeof(T)) % E);
  const int head = mis ? min(n, E - mis) : 0;
  for (int j = threadIdx.x; j < head; j += kST) fn(j, load_x<T>(x, j));
  const int nv = (n - head) / E;
  const uint4* vp = reinterpret_cast<const uint4*>(x + head);
  int v = threadIdx.x;
  for (; v + kST < nv; v += 2 * kST) {  // two vectors in flight a thread
    const uint4 q0 = __ldg(vp + v), q1 = __ldg(vp + v + kST);
#pragma unroll
    for (int e = 0; e < E; ++e) fn(head + v * E + e, vec_elem<T>(q0, e));
#pragma unroll
    for (int e = 0; e < E; ++e) fn(head + (v + kST) * E + e, vec_elem<T>(q1, e));
  }
  if (v < nv) {
    const uint4 q = __ldg(vp + v);
#pragma unroll
    for (int e = 0; e < E; ++e) fn(head + v * E + e, vec_elem<T>(q, e));
  }
  for (int j = head + nv * E + threadIdx.x; j < n; j += kST) fn(j, load_x<T>(x, j));
}

// The r-th largest of the distinct keys keys[0, n) (1 <= r <= n): byte-wise
// radix selection, most significant byte first, stopping once one key is left.
__device__ uint64_t select_kth_desc(const uint64_t* keys, int n, int r, ShardSmem& s) {
  uint64_t prefix = 0ull, mask = 0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += kST) s.hist[b] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kST) {
      const uint64_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&s.hist[(k >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bin_desc(s.hist, r, &s.bi[0], &s.bi[1]);
    __syncthreads();
    const int b = max(s.bi[0], 0);  // (r never exceeds the keys matching the prefix)
    const unsigned int in_bin = s.hist[b];
    prefix |= (uint64_t)b << shift;
    mask |= 0xFFull << shift;
    r = s.bi[1];
    if (in_bin == 1u) {
      for (int i = threadIdx.x; i < n; i += kST)
        if ((keys[i] & mask) == prefix) s.found = keys[i];
      __syncthreads();
      return s.found;
    }
    __syncthreads();
  }
  return prefix;
}

// The m largest of the distinct keys keys[0, n) (m <= VT_SHARD_MAX_K), sorted
// descending into s.sel[0, m): a selection of the m-th, a gather, a small sort.
__device__ void sorted_top(const uint64_t* keys, int n, int m, ShardSmem& s) {
  m = min(m, n);
  const uint64_t kmin = (m > 0 && n > m) ? select_kth_desc(keys, n, m, s) : 0ull;
  int P2 = 64;
  while (P2 < m) P2 <<= 1;
  if (threadIdx.x == 0) s.nsel = 0;
  for (int i = threadIdx.x; i < P2; i += kST) s.sel[i] = 0ull;
  __syncthreads();
  if (m > 0)
    for (int i = threadIdx.x; i < n; i += kST) {
      const uint64_t k = keys[i];
      if (k >= kmin) s.sel[atomicAdd(&s.nsel, 1)] = k;
    }
  __syncthreads();
  smem_sort_desc<kST>(s.sel, P2);
}

// ---------------------------------------------------------------------------
// partials: one CTA per row of the shard
// ---------------------------------------------------------------------------
// The shard's K largest elements, exactly, when the quick threshold let more
// than kShardCand elements through (a flat row, heavy ties, masked columns):
// a most-significant-digit radix select over the order-preserving bits of z_t,
// eight bits a pass, gives the K-th largest value; then one pass collects the
// elements above it and, in index order, the lowest-index elements equal to
// it.  Leaves the K records unsorted in s.keys[0, K).
template <typename T>
__device__ void shard_exact_top(const ShardArgs& a, const T* x, float inv_t, ShardSmem& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0u, mask = 0u;
  int r = a.K;  // rank of the wanted value among the elements matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kST) s.hist[i] = 0;
    __syncthreads();
    scan_elems<T>(x, a.Vs, [&](int, float xv) {
      const uint32_t o = ord_key(__fmul_rn(xv, inv_t));
      if ((o & mask) == prefix) atomicAdd(&s.hist[(o >> shift) & 255u], 1u);
    });
    __syncthreads();
    if (tid == 0) {
      int above = 0, b = 255;
      for (; b > 0 && above + (int)s.hist[b] < r; --b) above += (int)s.hist[b];
      s.bi[0] = b;
      s.bi[1] = r - above;
    }
    __syncthreads();
    prefix |= (uint32_t)s.bi[0] << shift;
    mask |= 255u << shift;
    r = s.bi[1];
    __syncthreads();
  }
  // K - r elements lie strictly above the K-th largest value; r ties are taken
  const int g = a.K - r;
  if (tid == 0) {
    s.count = 0;
    s.ties = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.Vs; base += kST) {
    const int j = base + tid;
    bool tie = false;
    if (j < a.Vs) {
      const float z = __fmul_rn(load_x<T>(x, j), inv_t);
      const uint32_t o = ord_key(z);
      if (o > prefix) s.keys[atomicAdd(&s.count, 1)] = elem_key(z, (uint32_t)(a.v0 + j));
      tie = o == prefix;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, tie);
    if (lane == 0) s.wt[warp] = __popc(bal);
    __syncthreads();
    int rank = s.ties + __popc(bal & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) rank += s.wt[w];
    if (tie && rank < r) s.keys[g + rank] = elem_key(key_value(prefix), (uint32_t)(a.v0 + j));
    __syncthreads();
    if (tid == 0)
      for (int w = 0; w < kSW; ++w) s.ties += s.wt[w];
    __syncthreads();
  }
}

template <typename T>
__global__ void __launch_bounds__(kST) shard_partials_kernel(const ShardArgs a) {
  __shared__ ShardSmem s;
  const int row = blockIdx.x, tid = threadIdx.x;
  const T* x = reinterpret_cast<const T*>(a.logits) + (int64_t)row * a.ld;
  const float inv_t = a.params[row].inv_t;
  // the shard's maximum, its lowest global index, and each thread's maximum
  float tmax = -INFINITY;
  int tj = INT_MAX;
  bool bad = false;
  scan_elems<T>(x, a.Vs, [&](int j, float xv) {
    const float z = __fmul_rn(xv, inv_t);
    bad |= (z != z) || z == INFINITY;
    if (z > tmax) {
      tmax = z;
      tj = a.v0 + j;
    }
  });
  s.tm[tid] = tmax;
  float m = tmax, zz = 0.f;
  int mj = tj;
  sblock_argmax(m, mj, zz, s);
  const int anybad = __syncthreads_or(bad);
  uint8_t* out = reinterpret_cast<uint8_t*>(a.part) + (size_t)row * a.part_bytes;
  if (anybad) {  // NaN or +inf: the merge reports the row as non-finite
    if (tid == 0) {
      ShardHead h{};
      h.m_t = m;
      h.s = 0.f;
      h.argj = mj;
      h.info = 1u << 30;
      h.wscore = -INFINITY;
      h.wj = INT_MAX;
      *reinterpret_cast<ShardHead*>(out) = h;
    }
    return;
  }
  // a lower bound of the shard's K-th largest: the K-th largest thread maximum
  // (at least K elements are >= it); -inf when fewer than K threads hold one
  if (tid == 0) {
    s.bf[3] = -INFINITY;
    s.count = 0;
  }
  __syncthreads();
  {
    const float v = s.tm[tid];
    int rank = 0;
    for (int u = 0; u < kST; ++u) {
      const float w = s.tm[u];
      rank += (w > v) || (w == v && u < tid);
    }
    if (rank == a.K - 1 && v > -INFINITY) s.bf[3] = v;
  }
  __syncthreads();
  const float tau = s.bf[3];
  // the sum of exponentials against m, and the elements at or above tau
  float sum = 0.f;
  const bool finite_max = m > -INFINITY;
  const float nh = __fmul_rn(-m, kLog2e);
  const float nl = finite_max ? __fmaf_rn(-m, kLog2e, -nh) : 0.f;
  // rows without a filter: the shard's Gumbel winner over its finite elements,
  // with the noise of the global (row, column) [the draw composes across
  // shards as an argmax], its finite count and its last finite element
  const bool unf = unfiltered_row(a.params[row], a.V);
  const uint64_t key = unf ? row_key(a.seeds[row], row) : 0ull;
  float ws = -INFINITY, wz = 0.f;
  int wj = INT_MAX;
  uint32_t nfin = 0u;
  unsigned long long last = 0ull;
  scan_elems<T>(x, a.Vs, [&](int j, float xv) {
    const float z = __fmul_rn(xv, inv_t);
    if (finite_max) sum += ex2_approx(__fadd_rn(__fmaf_rn(z, kLog2e, nh), nl));
    if (z >= tau) {
      const int pos = atomicAdd(&s.count, 1);
      if (pos < kShardCand) s.keys[pos] = elem_key(z, (uint32_t)(a.v0 + j));
    }
    if (unf && z > -INFINITY) {
      const int gj = a.v0 + j;
      ++nfin;
      const unsigned long long nk = ~elem_key(z, (uint32_t)gj);
      last = nk > last ? nk : last;
      const uint32_t b = noise_bits(key, gj);
      if (ws == -INFINITY || may_beat(z, ws, b)) {
        const float sc = gumbel_score(z, b);
        if (pair_better(sc, gj, ws, wj)) {
          ws = sc;
          wj = gj;
          wz = z;
        }
      }
    }
  });
  sum = sblock_sum(sum, s);
  if (unf) {
    sblock_argmax(ws, wj, wz, s);
    nfin = (uint32_t)sblock_sum_u64((unsigned long long)nfin, s);
    last = sblock_max_u64(last, s);
  }
  int n = s.count;
  __syncthreads();
  if (n > kShardCand) {
    shard_exact_top<T>(a, x, inv_t, s);
    n = a.K;
  }
  const int w = min(n, a.K);
  sorted_top(s.keys, n, w, s);
  uint64_t* rec = reinterpret_cast<uint64_t*>(out + sizeof(ShardHead));
  for (int i = tid; i < w; i += kST) rec[i] = s.sel[i];
  if (tid == 0) {
    ShardHead h{};
    h.m_t = m;
    h.s = sum;
    h.argj = mj;
    h.info = (uint32_t)w;
    h.wscore = ws;
    h.wj = wj;
    h.wz = wz;
    h.nfin = nfin;
    h.last = last;
    *reinterpret_cast<ShardHead*>(out) = h;
  }
}

// ---------------------------------------------------------------------------
// merge: one CTA per row, over the S shards' partials
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kST) shard_merge_kernel(const ShardArgs a) {
  __shared__ ShardSmem s;
  const int row = blockIdx.x, tid = threadIdx.x;
  const RowParams P = a.params[row];
  const int n = a.n_logprobs;
  // the row's statistics
  if (tid == 0) {
    float mt = -INFINITY, sm = 0.f, ws = -INFINITY, wz = 0.f;
    int argj = INT_MAX, bad = 0, total = 0, wj = INT_MAX;
    unsigned int nfin = 0u;
    unsigned long long last = 0ull;
    for (int sh = 0; sh < a.S; ++sh) {
      const uint8_t* in = reinterpret_cast<const uint8_t*>(a.part) +
                          ((size_t)sh * a.B + row) * a.part_bytes;
      const ShardHead h = *reinterpret_cast<const ShardHead*>(in);
      if (pair_better(h.m_t, h.argj, mt, argj) && h.m_t > -INFINITY) argj = h.argj;
      lse_combine(mt, sm, h.m_t, h.s, kLog2e);
      bad |= (h.info >> 30) & 1u;
      total += (int)(h.info & 0xFFFFu);
      if (h.wj != INT_MAX && pair_better(h.wscore, h.wj, ws, wj)) {
        ws = h.wscore;
        wj = h.wj;
        wz = h.wz;
      }
      nfin += h.nfin;
      last = h.last > last ? h.last : last;
    }
    s.w_score = ws;
    s.w_j = wj;
    s.w_z = wz;
    s.nfin_all = nfin;
    s.last_all = last;
    s.bf[0] = mt;
    s.bf[1] = sm;
    s.bi[0] = argj;
    s.bi[1] = bad || mt == INFINITY;
    s.bi[2] = total;
    s.bi[3] = total > kShardCand;  // the host keeps S * K within kShardCand
  }
  __syncthreads();
  const float m_t = s.bf[0], S = s.bf[1];
  const int argj = s.bi[0], bad = s.bi[1], ovf = s.bi[3];
  const int total = min(s.bi[2], kShardCand);
  const float lnS = logf(S);
  __syncthreads();
  const int status = bad ? kRowNonfinite : (m_t == -INFINITY ? kRowEmpty : kRowOk);
  if (status != kRowOk || ovf) {
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
      if (ovf) atomicOr(a.err_word, kErrInternal);
    }
    return;
  }
  // the union of the shards' records, in the order (z_t desc, index asc)
  {
    int off = 0;
    for (int sh = 0; sh < a.S; ++sh) {
      const uint8_t* in = reinterpret_cast<const uint8_t*>(a.part) +
                          ((size_t)sh * a.B + row) * a.part_bytes;
      const int w = (int)(reinterpret_cast<const ShardHead*>(in)->info & 0xFFFFu);
      const uint64_t* rec = reinterpret_cast<const uint64_t*>(in + sizeof(ShardHead));
      for (int i = tid; i < w && off + i < kShardCand; i += kST) s.keys[off + i] = rec[i];
      off += w;
    }
  }
  __syncthreads();
  // finite records, and min-p survivors (order-independent counts)
  const bool greedy = (P.flags & kRowGreedy) != 0;
  const bool minp = (P.flags & kRowMinP) != 0;
  int fin = 0, pass = 0;
  for (int i = tid; i < total; i += kST) {
    const float z = key_z(s.keys[i]);
    fin += z > -INFINITY;
    pass += minp && z > -INFINITY && minp_pass(z, m_t, P.log_min_p);
  }
  fin = (int)sblock_sum_u64((unsigned long long)fin, s);
  const int L1 = minp ? (int)sblock_sum_u64((unsigned long long)pass, s) : fin;
  // the leading records in the order (z_t desc, index asc): the top-n and the
  // top-k survivors
  const int L2 = (greedy || unfiltered_row(P, a.V)) ? 0 : min(P.top_k, L1);
  sorted_top(s.keys, total, max(n, L2), s);
  // top-n: the first n records
  for (int t = tid; t < n; t += kST) {
    if (t < total) {
      const uint64_t k = s.sel[t];
      a.out_topk_ids[(int64_t)row * n + t] = (int)key_idx(k);
      a.out_topk_logprobs[(int64_t)row * n + t] = (key_z(k) - m_t) - lnS;
    } else {
      a.out_topk_ids[(int64_t)row * n + t] = -1;
      a.out_topk_logprobs[(int64_t)row * n + t] = -INFINITY;
    }
  }
  if (unfiltered_row(P, a.V)) {
    // every finite element kept: the best of the shards' Gumbel winners
    if (tid == 0) {
      const uint64_t lk = ~s.last_all;
      a.out_tokens[row] = s.w_j;
      if (a.out_logprobs) a.out_logprobs[row] = (s.w_z - m_t) - lnS;
      a.row_status[row] = kRowOk;
      a.dbg_kth_value[row] = key_z(lk);
      a.dbg_kth_index[row] = (int)key_idx(lk);
      a.dbg_kept[row] = (int)s.nfin_all;
      a.seeds[row] += kSeedStep;
    }
    return;
  }
  int tok = argj, L3 = 1;
  float ztok = m_t;
  if (!greedy) {
    // min-p, then top-k, then top-p over the top-k survivors renormalised
    L3 = L2;
    if (P.flags & kRowTopP) {
      // exclusive prefix masses in 2^-43 fixed point; kept while <= p * W
      unsigned long long mine = 0ull;
      const int per = (L2 + kST - 1) / kST;
      const int i0 = min(L2, tid * per), i1 = min(L2, i0 + per);
      for (int i = i0; i < i1; ++i) mine += mass_fixed(key_z(s.sel[i]), m_t);
      // exclusive scan over the threads (serial in warp 0: at most 256 terms)
      s.ru[0] = 0ull;
      __syncthreads();
      __shared__ unsigned long long part[kST];
      part[tid] = mine;
      __syncthreads();
      if (tid == 0) {
        unsigned long long run = 0ull;
        for (int t = 0; t < kST; ++t) {
          const unsigned long long v = part[t];
          part[t] = run;
          run += v;
        }
        s.ru[1] = run;
      }
      __syncthreads();
      const unsigned long long W = s.ru[1];
      const unsigned long long Tm = (unsigned long long)((double)W * (double)P.top_p);
      unsigned long long run = part[tid];
      int kept = 0;
      for (int i = i0; i < i1; ++i) {
        if (run <= Tm) ++kept;
        run += mass_fixed(key_z(s.sel[i]), m_t);
      }
      L3 = max(1, (int)sblock_sum_u64((unsigned long long)kept, s));
    }
    // the Gumbel-max draw over the kept records, noise keyed by the global row
    // and column
    const uint64_t key = row_key(a.seeds[row], row);
    float bs = -INFINITY, bz = 0.f;
    int bj = INT_MAX;
    for (int i = tid; i < L3; i += kST) {
      const uint64_t k = s.sel[i];
      const int j = (int)key_idx(k);
      const float z = key_z(k);
      const float sc = gumbel_score_inl(z, noise_bits(key, j));
      if (pair_better(sc, j, bs, bj)) {
        bs = sc;
        bj = j;
        bz = z;
      }
    }
    sblock_argmax(bs, bj, bz, s);
    tok = bj;
    ztok = bz;
  }
  if (tid == 0) {
    a.out_tokens[row] = tok;
    if (a.out_logprobs) a.out_logprobs[row] = (ztok - m_t) - lnS;
    a.row_status[row] = kRowOk;
    const uint64_t kk = greedy ? 0ull : s.sel[L3 - 1];
    a.dbg_kth_value[row] = greedy ? m_t : key_z(kk);
    a.dbg_kth_index[row] = greedy ? tok : (int)key_idx(kk);
    a.dbg_kept[row] = L3;
    a.seeds[row] += kSeedStep;
  }
}

}  // namespace

int64_t shard_part_bytes(int K) { return (int64_t)sizeof(ShardHead) + 8 * (int64_t)K; }

cudaError_t launch_shard_partials(const ShardArgs& a, int dtype, cudaStream_t stream) {
  if (a.B < 1) return cudaSuccess;
  if (dtype == 0)
    shard_partials_kernel<float><<<a.B, kST, 0, stream>>>(a);
  else
    shard_partials_kernel<uint16_t><<<a.B, kST, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_shard_merge(const ShardArgs& a, cudaStream_t stream) {
  if (a.B < 1) return cudaSuccess;
  shard_merge_kernel<<<a.B, kST, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace vt
