// vt_counts.cu -- per-row token-count tables for the occurrence penalties.
//
// The penalties of the TensorRT-LLM "Sampling" page use c_j, the number of
// times token j occurs in the prompt plus everything generated so far; the
// first prompt_ignore_length prompt tokens count for the repetition penalty
// only.  At a counts reset each row's raw occurrences (prompt then output,
// CSR; each (id << 1) | ignored) are sorted in shared memory and run-length
// encoded into a table of distinct ids in increasing order, each with the
// number of its occurrences that count for presence and frequency (possibly
// 0: an id in the table is seen, for repetition).  The sampling kernel reads
// the slice of the table that falls in each CTA's part of the row and
// appends drawn tokens.
#include "vt_device.cuh"
#include "vt_kernels.h"

#include <climits>

namespace vt {
namespace {

constexpr int kCountThreads = 1024;

__global__ void __launch_bounds__(kCountThreads)
    build_counts_kernel(const int32_t* raw, const int64_t* offs, int2* hist, int32_t* hist_len,
                        int32_t hist_cap) {
  extern __shared__ int32_t keys[];
  __shared__ int warp_tot[kCountThreads / 32];
  __shared__ int warp_off[kCountThreads / 32];
  const int row = blockIdx.x;
  const int64_t a = offs[row];
  const int len = (int)(offs[row + 1] - a);
  int P2 = 1;
  while (P2 < len) P2 <<= 1;
  for (int i = threadIdx.x; i < P2; i += kCountThreads) keys[i] = i < len ? raw[a + i] : INT_MAX;
  __syncthreads();
  // bitonic sort, ascending
  for (int k = 2; k <= P2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P2; i += kCountThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int x = keys[i], y = keys[ixj];
          const bool up = (i & k) == 0;
          if (up ? (x > y) : (x < y)) {
            keys[i] = y;
            keys[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  // run starts in contiguous chunks, block scan of the chunk counts
  const int per = (len + kCountThreads - 1) / kCountThreads;
  const int i0 = min(len, (int)threadIdx.x * per), i1 = min(len, i0 + per);
  int starts = 0;
  for (int i = i0; i < i1; ++i) starts += (i == 0 || (keys[i] >> 1) != (keys[i - 1] >> 1));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = starts;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int w = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += w;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int t = warp_tot[lane];
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += w;
    }
    warp_off[lane] = ti - t;
    if (lane == 31) hist_len[row] = ti;
  }
  __syncthreads();
  int pos = warp_off[warp] + inc - starts;
  int2* out = hist + (int64_t)row * hist_cap;
  for (int i = i0; i < i1; ++i) {
    if (i == 0 || (keys[i] >> 1) != (keys[i - 1] >> 1)) {
      // the id's counted occurrences (flag 0) sort first: they end at the
      // first key above (id << 1) (binary search)
      int lo = i, hi = len;
      const int key = keys[i] & ~1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (keys[mid] > key) hi = mid; else lo = mid + 1;
      }
      out[pos++] = make_int2(key >> 1, lo - i);
    }
  }
}

}  // namespace

cudaError_t launch_build_counts(const int32_t* raw, const int64_t* offs, int max_len, int B,
                                int2* hist, int32_t* hist_len, int32_t hist_cap,
                                cudaStream_t stream) {
  if (B <= 0) return cudaSuccess;
  int P2 = 1;
  while (P2 < max_len) P2 <<= 1;
  const size_t smem = (size_t)P2 * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(build_counts_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  build_counts_kernel<<<B, kCountThreads, smem, stream>>>(raw, offs, hist, hist_len, hist_cap);
  return cudaGetLastError();
}

}  // namespace vt
