// vt_noalloc.cu -- vt_sample_noalloc: one sampling step that allocates nothing.
//
// Some callers may not allocate device memory at all.  A serving engine that
// sizes its KV-cache pool at start-up to fill nearly all of device memory
// leaves nothing for a library's own buffers, and often forbids later driver
// allocations outright.  A host whose device memory belongs to a framework's
// caching allocator cannot have a library take memory behind that allocator's
// back.  A decode loop with a latency budget keeps cudaMalloc and cudaFree
// out of it, because cudaFree waits for the whole device.  Such a caller
// cannot create a vt_sampler handle, since vt_sampler_create allocates every
// buffer the handle will use.
//
// This entry point therefore works in one fixed device array that this file
// defines, of VT_NOALLOC_SCRATCH_BYTES.  Its address is looked up once per
// device, with that device current, through cudaGetSymbolAddress.  Every call
// on a device works in the same array.  Two calls whose GPU work overlaps,
// because they run on different streams or come from different host threads,
// race on it.  Calls issued on one stream, one after the other, do not.
#include "vt_sampler.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "vt_device.cuh"
#include "vt_kernels.h"

// Scratch layout (byte offsets).  Rows beyond VT_NOALLOC_MAX_BATCH do not fit.
namespace {

constexpr int kMaxRows = VT_NOALLOC_MAX_BATCH;
constexpr size_t kOffParams = 0;                                        // RowParams[rows]
constexpr size_t kOffSeeds = kOffParams + kMaxRows * sizeof(vt::RowParams);  // uint64[rows]
constexpr size_t kOffHistLen = kOffSeeds + kMaxRows * sizeof(uint64_t);  // int32[rows], zero
constexpr size_t kOffStatus = kOffHistLen + kMaxRows * sizeof(int32_t);   // int32[rows]
constexpr size_t kOffKthV = kOffStatus + kMaxRows * sizeof(int32_t);      // float[rows]
constexpr size_t kOffKthI = kOffKthV + kMaxRows * sizeof(float);          // int32[rows]
constexpr size_t kOffKept = kOffKthI + kMaxRows * sizeof(int32_t);        // int32[rows]
constexpr size_t kOffSlow = kOffKept + kMaxRows * sizeof(int32_t);        // SlowRow[rows]
constexpr size_t kOffSlowList = kOffSlow + kMaxRows * sizeof(vt::SlowRow);  // int32[rows]
constexpr size_t kOffSlowCtl = kOffSlowList + kMaxRows * sizeof(int32_t);   // uint32[2], zero
constexpr size_t kOffErr = kOffSlowCtl + 16;                               // int32, zero
static_assert(kOffErr - kOffSlowCtl >= 3 * sizeof(uint32_t), "three hand-over words");
constexpr size_t kUsedBytes = kOffErr + 256;
static_assert(kUsedBytes <= VT_NOALLOC_SCRATCH_BYTES, "scratch layout exceeds its array");
static_assert(kOffSeeds % 16 == 0 && kOffSlow % 16 == 0 && kOffErr % 16 == 0,
              "scratch fields stay aligned");

}  // namespace

static __device__ __align__(256) unsigned char vt_noalloc_scratch[VT_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kUploadChunk = 64;  // rows of parameters staged on the host stack at once

struct DeviceSlot {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of vt_noalloc_scratch
  int num_sms = 0;
  size_t smem_optin = 0;
  // launch plans already prepared on this device, by (B, V, dtype): planning
  // sets kernel attributes and queries occupancy, which a decode loop should
  // not pay on every step (host memory only)
  std::map<std::tuple<int, int, int>, vt::LaunchPlan> plans;
};

std::mutex g_setup_mutex;
DeviceSlot g_slots[kMaxDevices];

int fail(char* errbuf, int32_t errlen, int code, const char* fmt, ...) {
  if (errbuf && errlen > 0) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(errbuf, (size_t)errlen, fmt, ap);
    va_end(ap);
  }
  return code;
}

// Make `dev` current for the duration of the call.
struct CurrentDevice {
  int prev = -1;
  bool ok = true;
  explicit CurrentDevice(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~CurrentDevice() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Once per device (the device is current): check the architecture, look up
// the scratch address and read the limits the launch plan needs.  A failed
// set-up is not remembered, so a later call tries again.
int setup_device(int dev, DeviceSlot** out, char* errbuf, int32_t errlen) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0, optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
      return fail(errbuf, errlen, VT_ERR_CUDA, "device %d attributes: %s", dev,
                  cudaGetErrorString(e));
    if (!(major == 10 && minor == 3))
      return fail(errbuf, errlen, VT_ERR_CUDA, "device %d is sm_%d%d; the library is built for sm_103a",
                  dev, major, minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, vt_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(errbuf, errlen, VT_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s",
                  cudaGetErrorString(e));
    s.scratch = static_cast<unsigned char*>(p);
    s.num_sms = sms;
    s.smem_optin = (size_t)optin;
    s.ready = true;
  }
  *out = &s;
  return VT_OK;
}

}  // namespace

extern "C" int vt_sample_noalloc(int32_t device, const void* logits, int32_t dtype, int32_t B,
                                 int32_t V, int64_t ld, const float* temperature,
                                 const int32_t* top_k, const float* top_p, const float* min_p,
                                 const uint64_t* seed, int32_t num_logprobs, int32_t* out_tokens,
                                 float* out_logprobs, int32_t* out_topk_ids,
                                 float* out_topk_logprobs, int32_t* row_status,
                                 int32_t synchronize, void* stream, char* errbuf,
                                 int32_t errbuf_len) {
  if (errbuf && errbuf_len > 0) errbuf[0] = '\0';
  // ---- sizes and arguments: all checked before any CUDA call ----
  if (B > kMaxRows)
    return fail(errbuf, errbuf_len, VT_ERR_CAPACITY,
                "B=%d rows exceed the no-allocation limit of %d rows (VT_NOALLOC_MAX_BATCH)", B,
                kMaxRows);
  if (B < 1) return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
  if (device < 0 || device >= kMaxDevices)
    return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "device %d out of range", device);
  if (dtype != VT_DTYPE_F32 && dtype != VT_DTYPE_BF16)
    return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (V > (1 << 20))
    return fail(errbuf, errbuf_len, VT_ERR_CAPACITY, "V=%d exceeds 1048576", V);
  if (V < 1 || ld < V)
    return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "need 1 <= V <= ld (V=%d, ld=%lld)", V,
                (long long)ld);
  if (num_logprobs < 0 || num_logprobs > 32)
    return fail(errbuf, errbuf_len, num_logprobs < 0 ? VT_ERR_INVALID_ARG : VT_ERR_CAPACITY,
                "num_logprobs=%d outside [0, 32]", num_logprobs);
  if (!logits || !out_tokens)
    return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "null logits or out_tokens");
  if (num_logprobs > 0 && (!out_topk_ids || !out_topk_logprobs))
    return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "top-n log-prob outputs are null");
  if (!temperature || !top_k || !top_p || !min_p || !seed)
    return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "null parameter array");
  for (int r = 0; r < B; ++r) {
    const float T = temperature[r], p = top_p[r], mp = min_p[r];
    if (!(T >= 0.0f) || !std::isfinite(T) || (T > 0.0f && !std::isfinite(1.0f / T)))
      return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "row %d: temperature %g out of range",
                  r, T);
    if (top_k[r] < 0) return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "row %d: top_k < 0", r);
    if (!(p >= 0.0f && p <= 1.0f))
      return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "row %d: top_p %g not in [0,1]", r, p);
    if (!(mp >= 0.0f && mp <= 1.0f))
      return fail(errbuf, errbuf_len, VT_ERR_INVALID_ARG, "row %d: min_p %g not in [0,1]", r, mp);
  }

  CurrentDevice guard(device);
  if (!guard.ok) return fail(errbuf, errbuf_len, VT_ERR_CUDA, "cannot select device %d", device);
  DeviceSlot* slot = nullptr;
  const int rc = setup_device(device, &slot, errbuf, errbuf_len);
  if (rc != VT_OK) return rc;

  const int es = dtype == VT_DTYPE_F32 ? 4 : 2;
  vt::LaunchPlan plan;
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    const auto key = std::make_tuple(B, V, dtype);
    auto it = slot->plans.find(key);
    if (it == slot->plans.end()) {
      vt::LaunchPlan fresh = vt::plan_sample(B, V, es, false, dtype, slot->num_sms);
      if (fresh.smem > slot->smem_optin)
        return fail(errbuf, errbuf_len, VT_ERR_CAPACITY,
                    "V=%d needs %zu B of shared memory per CTA", V, fresh.smem);
      e = vt::prepare_sample(fresh, dtype);
      if (e != cudaSuccess)
        return fail(errbuf, errbuf_len, VT_ERR_CUDA, "cannot prepare a %d-CTA cluster plan: %s",
                    fresh.cluster, cudaGetErrorString(e));
      it = slot->plans.emplace(key, fresh).first;
    }
    plan = it->second;
  }

  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* scr = slot->scratch;
  auto* d_params = reinterpret_cast<vt::RowParams*>(scr + kOffParams);
  auto* d_seeds = reinterpret_cast<uint64_t*>(scr + kOffSeeds);
  auto* d_hist_len = reinterpret_cast<int32_t*>(scr + kOffHistLen);
  auto* d_err = reinterpret_cast<int32_t*>(scr + kOffErr);

  // Per-row parameters, derived as vt_reset_params derives them (no
  // penalties), staged through a small host-stack buffer.  A copy from
  // pageable memory returns once the source has been read, so the buffer can
  // be reused for the next chunk.
  vt::RowParams hp[kUploadChunk];
  for (int r0 = 0; r0 < B; r0 += kUploadChunk) {
    const int m = B - r0 < kUploadChunk ? B - r0 : kUploadChunk;
    for (int i = 0; i < m; ++i) {
      const int r = r0 + i;
      const float T = temperature[r], p = top_p[r], mp = min_p[r];
      const int k = top_k[r];
      vt::RowParams& q = hp[i];
      std::memset(&q, 0, sizeof q);
      const bool greedy = T == 0.0f || k == 1 || p == 0.0f || mp == 1.0f;
      q.inv_t = greedy ? 1.0f : 1.0f / T;
      q.top_p = p;
      q.top_k = k;
      q.flags = greedy ? vt::kRowGreedy : 0u;
      if (p > 0.0f && p < 1.0f) q.flags |= vt::kRowTopP;
      if (mp > 0.0f && mp < 1.0f) q.flags |= vt::kRowMinP;
      q.presence = 0.0f;
      q.frequency = 0.0f;
      q.repetition = 1.0f;
      q.min_p = mp;
      q.log_min_p = (mp > 0.0f && mp < 1.0f) ? std::log((double)mp) : 0.0;
    }
    e = cudaMemcpyAsync(d_params + r0, hp, (size_t)m * sizeof(vt::RowParams),
                        cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
      return fail(errbuf, errbuf_len, VT_ERR_CUDA, "parameter upload: %s", cudaGetErrorString(e));
  }
  // The seeds go through the same kind of host-stack chunk, so that the call
  // has read the caller's array before it returns even when that array is
  // pinned (a copy straight from pinned memory would still be in flight).
  uint64_t hs[kUploadChunk];
  for (int r0 = 0; r0 < B && e == cudaSuccess; r0 += kUploadChunk) {
    const int m = B - r0 < kUploadChunk ? B - r0 : kUploadChunk;
    for (int i = 0; i < m; ++i) hs[i] = seed[r0 + i];
    e = cudaMemcpyAsync(d_seeds + r0, hs, (size_t)m * sizeof(uint64_t), cudaMemcpyHostToDevice,
                        st);
  }
  // What must start at zero: the rows' count-table lengths (no penalties, so
  // no table), the hand-over counters between the two kernels and the device
  // error word (the last three are contiguous).
  auto* d_slow_ctl = reinterpret_cast<uint32_t*>(scr + kOffSlowCtl);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_hist_len, 0, (size_t)B * sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_slow_ctl, 0, kOffErr + sizeof(int32_t) - kOffSlowCtl, st);
  if (e != cudaSuccess)
    return fail(errbuf, errbuf_len, VT_ERR_CUDA, "scratch set-up: %s", cudaGetErrorString(e));

  vt::SampleArgs a;
  std::memset(&a, 0, sizeof a);
  a.logits = logits;
  a.ld = ld;
  a.B = B;
  a.V = V;
  a.n_logprobs = num_logprobs;
  a.update_counts = 0;
  a.slice = plan.slice;
  a.aligned = ((uintptr_t)logits % 16 == 0) && (((uint64_t)ld * es) % 16 == 0);
  a.pen_smem = plan.pen_smem;
  a.off_gmax = plan.off_gmax;
  a.off_mrg = plan.off_mrg;
  a.off_bitmap = plan.off_bitmap;
  a.off_prefix = plan.off_prefix;
  a.params = d_params;
  a.seeds = d_seeds;
  a.decay = nullptr;  // no top-p decay on this path
  a.hist = nullptr;  // read only for rows with penalties or with update_counts
  a.hist_len = d_hist_len;
  a.hist_cap = 1;
  a.zside = nullptr;
  a.out_tokens = out_tokens;
  a.out_logprobs = out_logprobs;
  a.out_topk_ids = num_logprobs > 0 ? out_topk_ids : nullptr;
  a.out_topk_logprobs = num_logprobs > 0 ? out_topk_logprobs : nullptr;
  a.row_status = row_status ? row_status : reinterpret_cast<int32_t*>(scr + kOffStatus);
  a.dbg_kth_value = reinterpret_cast<float*>(scr + kOffKthV);
  a.dbg_kth_index = reinterpret_cast<int32_t*>(scr + kOffKthI);
  a.dbg_kept = reinterpret_cast<int32_t*>(scr + kOffKept);
  a.err_word = d_err;
  a.slow = reinterpret_cast<vt::SlowRow*>(scr + kOffSlow);
  a.slow_list = reinterpret_cast<int32_t*>(scr + kOffSlowList);
  a.slow_ctl = d_slow_ctl;
  a.trace = nullptr;
  a.trace_ctas = 0;
  e = vt::launch_sample(a, plan, dtype, st);
  if (e != cudaSuccess)
    return fail(errbuf, errbuf_len, VT_ERR_CUDA, "launch: %s", cudaGetErrorString(e));

  if (synchronize) {
    e = cudaStreamSynchronize(st);
    int32_t word = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&word, d_err, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
      return fail(errbuf, errbuf_len, VT_ERR_CUDA, "synchronise: %s", cudaGetErrorString(e));
    if (word & vt::kErrTimeout)
      return fail(errbuf, errbuf_len, VT_ERR_TIMEOUT, "a bounded device wait ran out");
    if (word != 0)
      return fail(errbuf, errbuf_len, VT_ERR_CUDA, "device error word 0x%x", word);
  }
  return VT_OK;
}
