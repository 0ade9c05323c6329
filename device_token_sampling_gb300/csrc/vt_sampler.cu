// vt_sampler.cu -- the C ABI of include/vt_sampler.h over the CUDA kernels.
//
// Host side only: argument validation, the reset-then-sample state machine
// (the Tenstorrent SamplingGenerator's reset_sampling_params / reset_seed /
// reset_prompt_tokens / reset_output_state / sample shape, with its rule that
// a sampler never reads state that was not reset), derived per-row values,
// pinned staging uploads, launch planning and launches.  Every device buffer
// and pinned buffer is allocated in vt_sampler_create; no other call allocates
// (the anti-pattern the vllm.cpp pull request records: a per-step cudaMalloc
// of the probabilities and a synchronising cudaFree).
#include "vt_sampler.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <map>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "vt_device.cuh"
#include "vt_kernels.h"

struct vt_sampler {
  vt_sampler_config cfg{};
  std::string err;
  // device state and scratch
  vt::RowParams* d_params = nullptr;
  uint64_t* d_seeds = nullptr;
  vt::DecayState* d_decay = nullptr;  // [max_batch] top-p decay state
  int2* d_hist = nullptr;
  int32_t* d_hist_len = nullptr;
  float* d_zside = nullptr;
  int32_t* d_raw = nullptr;
  int64_t* d_raw_offs = nullptr;
  int32_t* d_status = nullptr;
  float* d_kth_v = nullptr;
  int32_t* d_kth_i = nullptr;
  int32_t* d_kept = nullptr;
  int32_t* d_err = nullptr;
  vt::SlowRow* d_slow = nullptr;  // rows handed from the streaming to the selection kernel
  int32_t* d_slow_list = nullptr;  // [2][max_batch]: one list per launch pair
  uint32_t* d_slow_ctl = nullptr;  // [2][4]
  int32_t* d_rows = nullptr;       // [max_batch]: main rows, then side rows
  void* d_flat = nullptr;           // scratch of the flat kernels (bf16 rows up to max_vocab)
  size_t flat_bytes = 0;
  float2* d_probs_part = nullptr;  // (max, exp-sum) partials of the filtered distribution
  size_t probs_part_cap = 0;
  // the side stream: rows routed straight to the selection kernel run there,
  // beside the main stream's launches (fork and join through events)
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaEvent_t ev_launched = nullptr;  // every side CTA has begun
  bool launch_order = true;           // main rows wait for ev_launched (while it works)
  int n_main = 0, n_side = 0;
  int last_launches = 0;  // kernels the last vt_sample launched
  int last_pairs = 1;     // hand-over lists the last vt_sample used
  int path = 1;  // 1: the streaming kernel; 2: the flat kernels where they apply
  // pinned host staging
  vt::RowParams* h_params = nullptr;
  uint64_t* h_seeds = nullptr;
  vt::DecayState* h_decay = nullptr;
  int32_t* h_raw = nullptr;
  int64_t* h_raw_offs = nullptr;
  int32_t* h_err = nullptr;
  int32_t* h_rows = nullptr;
  cudaEvent_t ev_params = nullptr, ev_counts = nullptr;
  bool params_pending = false, counts_pending = false;
  // staging for vt_sample_host
  // host-memory calls: two staging slots; a step's logits are copied in on
  // io_copy while the previous step samples on the caller's stream
  struct IoSlot {
    void* logits = nullptr;
    int32_t* tokens = nullptr;
    float* lp = nullptr;
    int32_t* tid = nullptr;
    float* tlp = nullptr;
    cudaEvent_t copied = nullptr;  // its logits are on the device
    cudaEvent_t done = nullptr;    // its step and output copies are complete
    bool busy = false;
  };
  IoSlot io[2];
  size_t io_bytes = 0;
  cudaStream_t io_copy = nullptr;
  int io_next = 0;
  // host mirror of the state machine
  int params_B = 0;
  std::vector<uint32_t> row_flags;
  int counts_B = 0;
  int last_B = 0;
  cudaStream_t last_stream = nullptr;
  std::map<std::pair<std::pair<int, int>, std::pair<int, int>>, vt::LaunchPlan> plans;
  int num_sms = 0;
  cudaEvent_t phase_event = nullptr;    // debug: recorded between the two launches
  unsigned long long* trace = nullptr;  // debug phase trace (caller-owned)
  int64_t trace_ctas = 0;
};

namespace {


// Host-side fault injection for the failure-path tests, read at each call:
//   VT_FAULT_INJECT=alloc:<n>  the n-th device allocation of vt_sampler_create
//                              (0-based) fails as if the device were full;
//   VT_FAULT_INJECT=upload     the parameter upload of vt_reset_params fails.
// Nothing on the device is made to fault.
int fault_alloc_index() {
  const char* e = std::getenv("VT_FAULT_INJECT");
  if (e && std::strncmp(e, "alloc:", 6) == 0) return std::atoi(e + 6);
  return -1;
}
bool fault_upload() {
  const char* e = std::getenv("VT_FAULT_INJECT");
  return e && std::strcmp(e, "upload") == 0;
}

int set_err(vt_sampler* h, int code, const char* fmt, ...) {
  if (h) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    h->err = buf;
  }
  return code;
}

// Make the handle's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

#define VT_CK(h, expr)                                                                      \
  do {                                                                                      \
    cudaError_t e_ = (expr);                                                                \
    if (e_ != cudaSuccess)                                                                  \
      return set_err((h), VT_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));     \
  } while (0)

void free_all(vt_sampler* h) {
  auto dfree = [](void* p) {
    if (p) cudaFree(p);
  };
  auto hfree = [](void* p) {
    if (p) cudaFreeHost(p);
  };
  dfree(h->d_params);
  dfree(h->d_seeds);
  dfree(h->d_decay);
  dfree(h->d_hist);
  dfree(h->d_hist_len);
  dfree(h->d_zside);
  dfree(h->d_raw);
  dfree(h->d_raw_offs);
  dfree(h->d_status);
  dfree(h->d_kth_v);
  dfree(h->d_kth_i);
  dfree(h->d_kept);
  dfree(h->d_err);
  dfree(h->d_slow);
  dfree(h->d_slow_list);
  dfree(h->d_slow_ctl);
  dfree(h->d_rows);
  dfree(h->d_flat);
  dfree(h->d_probs_part);
  if (h->h_rows) cudaFreeHost(h->h_rows);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->ev_launched) cudaEventDestroy(h->ev_launched);
  if (h->side) cudaStreamDestroy(h->side);
  for (auto& slot : h->io) {
    dfree(slot.logits);
    dfree(slot.tokens);
    dfree(slot.lp);
    dfree(slot.tid);
    dfree(slot.tlp);
    if (slot.copied) cudaEventDestroy(slot.copied);
    if (slot.done) cudaEventDestroy(slot.done);
  }
  if (h->io_copy) cudaStreamDestroy(h->io_copy);
  hfree(h->h_params);
  hfree(h->h_seeds);
  hfree(h->h_decay);
  hfree(h->h_raw);
  hfree(h->h_raw_offs);
  hfree(h->h_err);
  if (h->ev_params) cudaEventDestroy(h->ev_params);
  if (h->ev_counts) cudaEventDestroy(h->ev_counts);
}

bool finite(float x) { return std::isfinite(x); }


}  // namespace

extern "C" {

const char* vt_status_string(int code) {
  switch (code) {
    case VT_OK: return "VT_OK";
    case VT_ERR_INVALID_ARG: return "VT_ERR_INVALID_ARG";
    case VT_ERR_STATE: return "VT_ERR_STATE";
    case VT_ERR_CAPACITY: return "VT_ERR_CAPACITY";
    case VT_ERR_CUDA: return "VT_ERR_CUDA";
    case VT_ERR_TIMEOUT: return "VT_ERR_TIMEOUT";
    default: return "VT_ERR_UNKNOWN";
  }
}

const char* vt_last_error(const vt_sampler* h) { return h ? h->err.c_str() : "null handle"; }

int vt_sampler_create(const vt_sampler_config* cfg, vt_sampler** out) {
  if (!cfg || !out) return VT_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->max_batch < 1 || cfg->max_batch > (1 << 20) || cfg->max_vocab < 1 ||
      cfg->max_vocab > (1 << 20) || cfg->max_logprobs < 0 || cfg->max_logprobs > 32 ||
      cfg->max_history < 0 || cfg->max_history > 32768 || cfg->device < 0)
    return VT_ERR_INVALID_ARG;
  vt_sampler* h = new (std::nothrow) vt_sampler();
  if (!h) return VT_ERR_CUDA;
  h->cfg = *cfg;
  DeviceGuard guard(cfg->device);
  auto bail = [&](int code) {
    free_all(h);
    delete h;
    return code;
  };
  if (!guard.ok) return bail(VT_ERR_CUDA);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return bail(VT_ERR_CUDA);
  if (!(prop.major == 10 && prop.minor == 3)) return bail(VT_ERR_CUDA);  // built for sm_103a only
  // the largest row must fit the shared-memory plan (16 CTAs per row at most)
  const vt::LaunchPlan worst = vt::plan_layout(cfg->max_vocab, 4, 16, true, true);
  if (worst.smem > (size_t)prop.sharedMemPerBlockOptin) return bail(VT_ERR_CAPACITY);
  h->num_sms = prop.multiProcessorCount;

  const size_t B = (size_t)cfg->max_batch;
  const size_t H = (size_t)(cfg->max_history > 0 ? cfg->max_history : 1);
  const size_t n = (size_t)cfg->max_logprobs;
  bool ok = true;
  const int fail_at = fault_alloc_index();
  int nalloc = 0;
  auto dal = [&](void** p, size_t bytes) {
    if (ok && (nalloc++ == fail_at || cudaMalloc(p, bytes) != cudaSuccess)) ok = false;
  };
  auto hal = [&](void** p, size_t bytes) {
    if (ok && cudaMallocHost(p, bytes) != cudaSuccess) ok = false;
  };
  dal((void**)&h->d_params, B * sizeof(vt::RowParams));
  dal((void**)&h->d_seeds, B * sizeof(uint64_t));
  dal((void**)&h->d_decay, B * sizeof(vt::DecayState));
  dal((void**)&h->d_hist, B * H * sizeof(int2));
  dal((void**)&h->d_hist_len, B * sizeof(int32_t));
  dal((void**)&h->d_zside, B * H * sizeof(float));
  dal((void**)&h->d_raw, B * H * sizeof(int32_t));
  dal((void**)&h->d_raw_offs, (B + 1) * sizeof(int64_t));
  dal((void**)&h->d_status, B * sizeof(int32_t));
  dal((void**)&h->d_kth_v, B * sizeof(float));
  dal((void**)&h->d_kth_i, B * sizeof(int32_t));
  dal((void**)&h->d_kept, B * sizeof(int32_t));
  dal((void**)&h->d_err, sizeof(int32_t));
  dal((void**)&h->d_slow, B * sizeof(vt::SlowRow));
  dal((void**)&h->d_slow_list, 2 * B * sizeof(int32_t));
  dal((void**)&h->d_slow_ctl, 8 * sizeof(uint32_t));
  dal((void**)&h->d_rows, B * sizeof(int32_t));
  // the flat kernels: slices of the widest row the handle takes
  {
    const vt::FlatPlan fp = vt::plan_flat(cfg->max_vocab);
    if (fp.C > 0) {
      h->flat_bytes = vt::flat_scratch_bytes((int)B, fp.C);
      dal(&h->d_flat, h->flat_bytes);
    }
  }
  // B rows of ceil(V / max range) + 1 splits, plus the splits that small
  // batches add to fill the GPU (plan_probs never asks for more)
  h->probs_part_cap = B * (size_t)((cfg->max_vocab + vt::kProbsMaxRange - 1) /
                                       vt::kProbsMaxRange + 1) +
                      (size_t)vt::kProbsCtasPerSm * h->num_sms;
  dal((void**)&h->d_probs_part, h->probs_part_cap * sizeof(float2));
  hal((void**)&h->h_rows, B * sizeof(int32_t));
  hal((void**)&h->h_params, B * sizeof(vt::RowParams));
  hal((void**)&h->h_seeds, B * sizeof(uint64_t));
  hal((void**)&h->h_decay, B * sizeof(vt::DecayState));
  hal((void**)&h->h_raw, B * H * sizeof(int32_t));
  hal((void**)&h->h_raw_offs, (B + 1) * sizeof(int64_t));
  hal((void**)&h->h_err, sizeof(int32_t));
  if (cfg->host_io) {
    h->io_bytes = B * (size_t)cfg->max_vocab * 4;
    for (auto& slot : h->io) {
      dal(&slot.logits, h->io_bytes);
      dal((void**)&slot.tokens, B * sizeof(int32_t));
      dal((void**)&slot.lp, B * sizeof(float));
      dal((void**)&slot.tid, B * (n ? n : 1) * sizeof(int32_t));
      dal((void**)&slot.tlp, B * (n ? n : 1) * sizeof(float));
      if (ok && (cudaEventCreateWithFlags(&slot.copied, cudaEventDisableTiming) != cudaSuccess ||
                 cudaEventCreateWithFlags(&slot.done, cudaEventDisableTiming) != cudaSuccess))
        ok = false;
    }
    if (ok && cudaStreamCreateWithFlags(&h->io_copy, cudaStreamNonBlocking) != cudaSuccess)
      ok = false;
  }
  if (!ok) return bail(VT_ERR_CUDA);
  if (cudaEventCreateWithFlags(&h->ev_params, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_counts, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_launched, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess)
    return bail(VT_ERR_CUDA);
  if (cudaMemset(h->d_hist_len, 0, B * sizeof(int32_t)) != cudaSuccess ||
      cudaMemset(h->d_err, 0, sizeof(int32_t)) != cudaSuccess ||
      cudaMemset(h->d_slow_ctl, 0, 8 * sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(h->d_seeds, 0, B * sizeof(uint64_t)) != cudaSuccess ||
      cudaMemset(h->d_status, 0, B * sizeof(int32_t)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return bail(VT_ERR_CUDA);
  *h->h_err = 0;
  h->row_flags.assign(B, 0u);
  *out = h;
  return VT_OK;
}

void vt_sampler_destroy(vt_sampler* h) {
  if (!h) return;
  DeviceGuard guard(h->cfg.device);
  if (h->last_stream) cudaStreamSynchronize(h->last_stream);
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
}

int vt_reset_params(vt_sampler* h, int32_t B, const float* temperature, const int32_t* top_k,
                    const float* top_p, const float* min_p, const float* presence,
                    const float* frequency, const float* repetition, const uint64_t* seed,
                    void* stream) {
  return vt_reset_params_ex(h, B, temperature, top_k, top_p, min_p, presence, frequency,
                            repetition, seed, nullptr, nullptr, nullptr, stream);
}

int vt_reset_params_ex(vt_sampler* h, int32_t B, const float* temperature, const int32_t* top_k,
                       const float* top_p, const float* min_p, const float* presence,
                       const float* frequency, const float* repetition, const uint64_t* seed,
                       const float* top_p_decay, const float* top_p_min,
                       const int32_t* top_p_reset_ids, void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  if (B < 1) return set_err(h, VT_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
  if (B > h->cfg.max_batch)
    return set_err(h, VT_ERR_CAPACITY, "B=%d exceeds max_batch=%d", B, h->cfg.max_batch);
  if (!temperature || !top_k || !top_p || !min_p || !presence || !frequency || !repetition ||
      !seed)
    return set_err(h, VT_ERR_INVALID_ARG, "null parameter array");
  for (int r = 0; r < B; ++r) {
    const float T = temperature[r], p = top_p[r], mp = min_p[r], rep = repetition[r];
    if (!(T >= 0.0f) || !finite(T) || (T > 0.0f && !finite(1.0f / T)))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: temperature %g out of range", r, T);
    if (top_k[r] < 0) return set_err(h, VT_ERR_INVALID_ARG, "row %d: top_k < 0", r);
    if (!(p >= 0.0f && p <= 1.0f))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: top_p %g not in [0,1]", r, p);
    if (!(mp >= 0.0f && mp <= 1.0f))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: min_p %g not in [0,1]", r, mp);
    if (!finite(presence[r]) || !finite(frequency[r]) || !finite(rep) || !(rep > 0.0f))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: penalties out of range", r);
    if (top_p_decay && !(top_p_decay[r] > 0.0f && top_p_decay[r] <= 1.0f))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: top_p_decay %g not in (0,1]", r,
                     top_p_decay[r]);
    if (top_p_min && !(top_p_min[r] > 0.0f && top_p_min[r] <= 1.0f))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: top_p_min %g not in (0,1]", r, top_p_min[r]);
    if (top_p_reset_ids && top_p_reset_ids[r] < -1)
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: top_p_reset_ids %d < -1", r,
                     top_p_reset_ids[r]);
  }
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return set_err(h, VT_ERR_CUDA, "cannot select device %d", h->cfg.device);
  cudaStream_t st = (cudaStream_t)stream;
  if (h->params_pending) {
    VT_CK(h, cudaEventSynchronize(h->ev_params));
    h->params_pending = false;
  }
  for (int r = 0; r < B; ++r) {
    const float T = temperature[r], p = top_p[r], mp = min_p[r];
    const int k = top_k[r];
    vt::RowParams rp;
    std::memset(&rp, 0, sizeof rp);
    const bool greedy = T == 0.0f || k == 1 || p == 0.0f || mp == 1.0f;
    rp.inv_t = greedy ? 1.0f : 1.0f / T;
    rp.top_p = p;
    rp.top_k = k;
    rp.flags = 0;
    if (greedy) rp.flags |= vt::kRowGreedy;
    if (p > 0.0f && p < 1.0f) rp.flags |= vt::kRowTopP;
    if (mp > 0.0f && mp < 1.0f) rp.flags |= vt::kRowMinP;
    if (presence[r] != 0.0f || frequency[r] != 0.0f || repetition[r] != 1.0f)
      rp.flags |= vt::kRowPenalty;
    // An active decay makes a sampled row a top-p row from its top_p (1 when
    // unset); the explicit greedy triggers take precedence.
    vt::DecayState ds;
    ds.p = p;
    ds.decay = top_p_decay ? top_p_decay[r] : 1.0f;
    ds.p_min = top_p_min ? top_p_min[r] : 1e-6f;
    ds.reset_id = top_p_reset_ids ? top_p_reset_ids[r] : -1;
    if (!greedy && ds.decay < 1.0f) rp.flags |= vt::kRowDecay;
    h->h_decay[r] = ds;
    rp.presence = presence[r];
    rp.frequency = frequency[r];
    rp.repetition = repetition[r];
    rp.min_p = mp;
    rp.log_min_p = (mp > 0.0f && mp < 1.0f) ? std::log((double)mp) : 0.0;
    h->h_params[r] = rp;
    h->h_seeds[r] = seed[r];
    h->row_flags[r] = rp.flags;
  }
  // Route the rows that will most likely need selection straight to the
  // selection kernel: sampled top-p rows without top-k and without penalties
  // (their nucleus is usually far beyond what one candidate pass gathers).
  // Used for bf16 calls over all B rows; main rows first, then side rows.
  auto to_side = [&](int r) {
    const uint32_t f = h->row_flags[r];
    return !(f & vt::kRowGreedy) && !(f & vt::kRowPenalty) && !(f & vt::kRowDecay) &&
           (f & vt::kRowTopP) && top_k[r] <= 1;
  };
  int nm = 0, ns = 0;
  for (int r = 0; r < B; ++r)
    if (!to_side(r)) h->h_rows[nm++] = r;
  for (int r = 0; r < B; ++r)
    if (to_side(r)) h->h_rows[nm + ns++] = r;
  // Clusters start in launch order, and the last ones may wait for room on
  // the SMs: the main rows go heaviest first (most candidates: top-k rows by
  // k, then the other filtered rows, greedy rows last), stable in row order.
  auto weight = [&](int r) {
    const uint32_t f = h->row_flags[r];
    if (f & vt::kRowGreedy) return 0;
    return top_k[r] > 1 ? top_k[r] : 1;
  };
  std::stable_sort(h->h_rows, h->h_rows + nm, [&](int x, int y) { return weight(x) > weight(y); });
  h->n_main = nm;
  h->n_side = ns;
  // A failed upload leaves the device parameters undefined: the handle then
  // counts as never reset (vt_sample returns VT_ERR_STATE until the next reset).
  h->params_B = 0;
  if (fault_upload()) return set_err(h, VT_ERR_CUDA, "parameter upload failed (injected fault)");
  VT_CK(h, cudaMemcpyAsync(h->d_params, h->h_params, (size_t)B * sizeof(vt::RowParams),
                           cudaMemcpyHostToDevice, st));
  VT_CK(h, cudaMemcpyAsync(h->d_seeds, h->h_seeds, (size_t)B * sizeof(uint64_t),
                           cudaMemcpyHostToDevice, st));
  VT_CK(h, cudaMemcpyAsync(h->d_decay, h->h_decay, (size_t)B * sizeof(vt::DecayState),
                           cudaMemcpyHostToDevice, st));
  VT_CK(h, cudaMemcpyAsync(h->d_rows, h->h_rows, (size_t)B * sizeof(int32_t),
                           cudaMemcpyHostToDevice, st));
  VT_CK(h, cudaEventRecord(h->ev_params, st));
  h->params_pending = true;
  h->params_B = B;
  h->last_stream = st;
  h->err.clear();
  return VT_OK;
}

int vt_reset_token_counts(vt_sampler* h, int32_t B, const int32_t* prompt_ids,
                          const int64_t* prompt_offsets, const int32_t* output_ids,
                          const int64_t* output_offsets, void* stream) {
  return vt_reset_token_counts_ex(h, B, prompt_ids, prompt_offsets, output_ids, output_offsets,
                                  nullptr, stream);
}

int vt_reset_token_counts_ex(vt_sampler* h, int32_t B, const int32_t* prompt_ids,
                             const int64_t* prompt_offsets, const int32_t* output_ids,
                             const int64_t* output_offsets, const int32_t* prompt_ignore_length,
                             void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  if (B < 1) return set_err(h, VT_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
  if (B > h->cfg.max_batch)
    return set_err(h, VT_ERR_CAPACITY, "B=%d exceeds max_batch=%d", B, h->cfg.max_batch);
  if (!prompt_offsets || !output_offsets)
    return set_err(h, VT_ERR_INVALID_ARG, "null offsets");
  if (prompt_offsets[0] != 0 || output_offsets[0] != 0)
    return set_err(h, VT_ERR_INVALID_ARG, "offsets must start at 0");
  int max_len = 0;
  for (int r = 0; r < B; ++r) {
    const int64_t np = prompt_offsets[r + 1] - prompt_offsets[r];
    const int64_t no = output_offsets[r + 1] - output_offsets[r];
    if (np < 0 || no < 0) return set_err(h, VT_ERR_INVALID_ARG, "row %d: decreasing offsets", r);
    if (np + no > h->cfg.max_history)
      return set_err(h, VT_ERR_CAPACITY, "row %d: %lld ids exceed max_history=%d", r,
                     (long long)(np + no), h->cfg.max_history);
    if ((np && !prompt_ids) || (no && !output_ids))
      return set_err(h, VT_ERR_INVALID_ARG, "null id array");
    max_len = (int)std::max<int64_t>(max_len, np + no);
  }
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return set_err(h, VT_ERR_CUDA, "cannot select device %d", h->cfg.device);
  cudaStream_t st = (cudaStream_t)stream;
  if (h->counts_pending) {
    VT_CK(h, cudaEventSynchronize(h->ev_counts));
    h->counts_pending = false;
  }
  // Each occurrence goes up as (id << 1) | ignored: ignored occurrences (the
  // first prompt_ignore_length prompt ids) count for repetition only.
  int64_t w = 0;
  h->h_raw_offs[0] = 0;
  for (int r = 0; r < B; ++r) {
    const int64_t skip = prompt_ignore_length && prompt_ignore_length[r] > 0
                             ? (int64_t)prompt_ignore_length[r]
                             : 0;
    for (int64_t i = prompt_offsets[r]; i < prompt_offsets[r + 1]; ++i) {
      const int32_t id = prompt_ids[i];
      if (id < 0 || id >= h->cfg.max_vocab)
        return set_err(h, VT_ERR_INVALID_ARG, "row %d: prompt id %d out of range", r, id);
      h->h_raw[w++] = (id << 1) | (i - prompt_offsets[r] < skip ? 1 : 0);
    }
    for (int64_t i = output_offsets[r]; i < output_offsets[r + 1]; ++i) {
      const int32_t id = output_ids[i];
      if (id < 0 || id >= h->cfg.max_vocab)
        return set_err(h, VT_ERR_INVALID_ARG, "row %d: output id %d out of range", r, id);
      h->h_raw[w++] = id << 1;
    }
    h->h_raw_offs[r + 1] = w;
  }
  if (w > 0)
    VT_CK(h, cudaMemcpyAsync(h->d_raw, h->h_raw, (size_t)w * sizeof(int32_t),
                             cudaMemcpyHostToDevice, st));
  VT_CK(h, cudaMemcpyAsync(h->d_raw_offs, h->h_raw_offs, (size_t)(B + 1) * sizeof(int64_t),
                           cudaMemcpyHostToDevice, st));
  VT_CK(h, vt::launch_build_counts(h->d_raw, h->d_raw_offs, max_len, B, h->d_hist,
                                   h->d_hist_len, h->cfg.max_history > 0 ? h->cfg.max_history : 1,
                                   st));
  VT_CK(h, cudaEventRecord(h->ev_counts, st));
  h->counts_pending = true;
  h->counts_B = B;
  h->last_stream = st;
  h->err.clear();
  return VT_OK;
}

static int sample_impl(vt_sampler* h, const void* logits, int32_t dtype, int32_t B, int32_t V,
                       int64_t ld, int32_t n, int32_t update_counts, int32_t* out_tokens,
                       float* out_logprobs, int32_t* out_topk_ids, float* out_topk_logprobs,
                       float* out_probs, int64_t ld_probs, cudaStream_t st) {
  if (h->params_B == 0) return set_err(h, VT_ERR_STATE, "vt_sample before vt_reset_params");
  if (B < 1 || B > h->params_B)
    return set_err(h, B < 1 ? VT_ERR_INVALID_ARG : VT_ERR_STATE,
                   "B=%d but parameters were reset for %d rows", B, h->params_B);
  if (dtype != VT_DTYPE_F32 && dtype != VT_DTYPE_BF16)
    return set_err(h, VT_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (V < 1 || ld < V) return set_err(h, VT_ERR_INVALID_ARG, "need 1 <= V <= ld");
  if (V > h->cfg.max_vocab)
    return set_err(h, VT_ERR_CAPACITY, "V=%d exceeds max_vocab=%d", V, h->cfg.max_vocab);
  if (n < 0 || n > h->cfg.max_logprobs)
    return set_err(h, n < 0 ? VT_ERR_INVALID_ARG : VT_ERR_CAPACITY,
                   "num_logprobs=%d outside [0, %d]", n, h->cfg.max_logprobs);
  if (!logits || !out_tokens) return set_err(h, VT_ERR_INVALID_ARG, "null logits or tokens");
  if (n > 0 && (!out_topk_ids || !out_topk_logprobs))
    return set_err(h, VT_ERR_INVALID_ARG, "top-k log-prob outputs are null");
  if ((update_counts && h->cfg.max_history == 0))
    return set_err(h, VT_ERR_CAPACITY, "update_counts needs max_history > 0");
  if (out_probs && ld_probs < V) return set_err(h, VT_ERR_INVALID_ARG, "ld_probs < V");
  for (int r = 0; r < B; ++r)
    if ((h->row_flags[r] & vt::kRowPenalty) && r >= h->counts_B)
      return set_err(h, VT_ERR_STATE, "row %d has penalties but its counts were never reset", r);
  const int es = dtype == VT_DTYPE_F32 ? 4 : 2;
  bool any_pen = false;
  for (int r = 0; r < B && !any_pen; ++r) any_pen = (h->row_flags[r] & vt::kRowPenalty) != 0;
  auto get_plan = [&](int rows, const vt::LaunchPlan** out) -> int {
    auto key = std::make_pair(std::make_pair(rows, V), std::make_pair(dtype, any_pen ? 1 : 0));
    auto it = h->plans.find(key);
    if (it == h->plans.end()) {
      vt::LaunchPlan plan = vt::plan_sample(rows, V, es, any_pen, dtype, h->num_sms);
      const cudaError_t e = vt::prepare_sample(plan, dtype);
      if (e != cudaSuccess)
        return set_err(h, VT_ERR_CUDA, "cannot prepare a %d-CTA cluster plan: %s", plan.cluster,
                       cudaGetErrorString(e));
      it = h->plans.emplace(key, plan).first;
    }
    *out = &it->second;
    return VT_OK;
  };
  auto make_args = [&](const vt::LaunchPlan& plan, int rows, const int32_t* row_list, int early,
                       int pair) {
    vt::SampleArgs a;
    std::memset(&a, 0, sizeof a);
    a.logits = logits;
    a.ld = ld;
    a.B = rows;
    a.V = V;
    a.rows = row_list;
    a.early = early;
    a.n_logprobs = n;
    // with the distribution exported, the counts are updated after it
    a.update_counts = update_counts && !out_probs ? 1 : 0;
    a.slice = plan.slice;
    a.aligned = ((uintptr_t)logits % 16 == 0) && (((uint64_t)ld * es) % 16 == 0);
    a.pen_smem = plan.pen_smem;
    a.off_gmax = plan.off_gmax;
    a.off_mrg = plan.off_mrg;
    a.off_bitmap = plan.off_bitmap;
    a.off_prefix = plan.off_prefix;
    a.params = h->d_params;
    a.seeds = h->d_seeds;
    a.decay = h->d_decay;
    a.hist = h->d_hist;
    a.hist_len = h->d_hist_len;
    a.hist_cap = h->cfg.max_history > 0 ? h->cfg.max_history : 1;
    a.zside = h->d_zside;
    a.out_tokens = out_tokens;
    a.out_logprobs = out_logprobs;
    a.out_topk_ids = out_topk_ids;
    a.out_topk_logprobs = out_topk_logprobs;
    a.row_status = h->d_status;
    a.dbg_kth_value = h->d_kth_v;
    a.dbg_kth_index = h->d_kth_i;
    a.dbg_kept = h->d_kept;
    a.err_word = h->d_err;
    a.slow = h->d_slow;
    a.slow_list = h->d_slow_list + (size_t)pair * h->cfg.max_batch;
    a.slow_ctl = h->d_slow_ctl + 4 * pair;
    // the phase trace is laid out by row (B rows of `plan.cluster` CTAs)
    a.trace = (h->trace && (int64_t)B * plan.cluster <= h->trace_ctas) ? h->trace : nullptr;
    a.trace_ctas = a.trace ? h->trace_ctas : 0;
    return a;
  };
  // bf16 calls without penalties or top-p decay on 16-byte aligned rows: the
  // flat kernels, then the selection kernel for the rows they hand over
  bool flat = false;
  vt::FlatPlan fplan{0, 0, 0};
  if (dtype == VT_DTYPE_BF16 && !any_pen && !out_probs && h->path == 2 && h->d_flat &&
      (uintptr_t)logits % 16 == 0 && ((uint64_t)ld * 2) % 16 == 0) {
    fplan = vt::plan_flat(V);
    bool decay = false;
    for (int r = 0; r < B && !decay; ++r) decay = (h->row_flags[r] & vt::kRowDecay) != 0;
    flat = fplan.C > 0 && !decay && vt::flat_scratch_bytes(B, fplan.C) <= h->flat_bytes;
  }
  if (flat) {
    const vt::LaunchPlan* plan = nullptr;
    const int rc = get_plan(B, &plan);
    if (rc != VT_OK) return rc;
    vt::SampleArgs sa = make_args(*plan, B, nullptr, 0, 0);
    sa.update_counts = 0;
    sa.trace = nullptr;
    sa.trace_ctas = 0;
    vt::FlatArgs fa;
    std::memset(&fa, 0, sizeof fa);
    fa.logits = logits;
    fa.ld = ld;
    fa.B = B;
    fa.V = V;
    fa.C = fplan.C;
    fa.L = fplan.L;
    fa.NV = fplan.NV;
    fa.n_logprobs = n;
    fa.params = h->d_params;
    fa.seeds = h->d_seeds;
    fa.out_tokens = out_tokens;
    fa.out_logprobs = out_logprobs;
    fa.out_topk_ids = out_topk_ids;
    fa.out_topk_logprobs = out_topk_logprobs;
    fa.row_status = h->d_status;
    fa.dbg_kth_value = h->d_kth_v;
    fa.dbg_kth_index = h->d_kth_i;
    fa.dbg_kept = h->d_kept;
    fa.slow = h->d_slow;
    fa.slow_list = sa.slow_list;
    fa.slow_ctl = sa.slow_ctl;
    fa.scratch = h->d_flat;
    VT_CK(h, vt::launch_flat(fa, st));
    if (h->phase_event) VT_CK(h, cudaEventRecord(h->phase_event, st));
    // rows the flat kernels hand over are rare (a top_k above their limit,
    // overflowing buffers): a few selection clusters, more for the former
    int certain = 0;
    for (int r = 0; r < B; ++r) {
      const int k = h->h_params[r].top_k;
      if (!(h->row_flags[r] & vt::kRowGreedy) && k > vt::kFlatKMax && k < V) ++certain;
    }
    VT_CK(h, vt::launch_select_handed(sa, *plan, dtype, st, certain + 4));
    h->last_launches = 7;
    h->last_pairs = 1;
    if (update_counts) {
      VT_CK(h, vt::launch_append(h->d_hist, h->d_hist_len, sa.hist_cap, out_tokens, h->d_status,
                                 B, st));
      h->last_launches += 1;
    }
    h->last_B = B;
    h->last_stream = st;
    h->err.clear();
    return VT_OK;
  }
  // other bf16 calls over every row split the rows between the two streams
  const bool split = dtype == VT_DTYPE_BF16 && B == h->params_B && h->n_side > 0 &&
                     h->n_main > 0;
  h->last_pairs = split ? 2 : 1;
  if (!split) {
    const vt::LaunchPlan* plan = nullptr;
    const int rc = get_plan(B, &plan);
    if (rc != VT_OK) return rc;
    const vt::SampleArgs a = make_args(*plan, B, nullptr, 0, 0);
    VT_CK(h, vt::launch_sample(a, *plan, dtype, st, h->phase_event));
    h->last_launches = 2;
  } else {
    // both launches keep the whole batch's slices, so that every row's sums
    // (and so its results) do not depend on how the rows are split
    const vt::LaunchPlan* pm = nullptr;
    const int rc = get_plan(B, &pm);
    if (rc != VT_OK) return rc;
    const vt::LaunchPlan* ps = pm;
    const vt::SampleArgs am = make_args(*pm, h->n_main, h->d_rows, 0, 0);
    const vt::SampleArgs as = make_args(*ps, h->n_side, h->d_rows + h->n_main, 1, 1);
    VT_CK(h, cudaEventRecord(h->ev_fork, st));
    VT_CK(h, cudaStreamWaitEvent(h->side, h->ev_fork, 0));
    // the side rows: the selection kernel alone, taking their statistics
    // itself (else the streaming kernel hands them over at once)
    // The side rows are the step's longest: the main rows' CTAs wait until
    // every side CTA has begun, so that the side ones never wait for room.
    // The order is a preference: where the launch-completion event or the
    // wait on it is refused (a profiler that serialises kernels refuses the
    // wait), the handle stops asking for it.  It is asked for only when every
    // side cluster fits on the GPU at once; else the main rows would wait for
    // the side kernel's last wave to begin.
    if (ps->own.cluster >= 1) {
      bool launched = false;
      if (h->launch_order && h->n_side <= ps->own.clusters) {
        if (vt::launch_select_own(as, *ps, dtype, h->side, h->ev_launched) == cudaSuccess) {
          launched = true;
          if (cudaStreamWaitEvent(st, h->ev_launched, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            h->launch_order = false;
          }
        } else {
          (void)cudaGetLastError();
          h->launch_order = false;
        }
      }
      if (!launched) VT_CK(h, vt::launch_select_own(as, *ps, dtype, h->side, nullptr));
    } else {
      VT_CK(h, vt::launch_sample(as, *ps, dtype, h->side, nullptr));
    }
    VT_CK(h, vt::launch_sample(am, *pm, dtype, st, h->phase_event));
    VT_CK(h, cudaEventRecord(h->ev_join, h->side));
    VT_CK(h, cudaStreamWaitEvent(st, h->ev_join, 0));
    h->last_launches = ps->own.cluster >= 1 ? 3 : 4;
  }
  if (out_probs) {
    vt::ProbsArgs pa;
    std::memset(&pa, 0, sizeof pa);
    pa.logits = logits;
    pa.ld = ld;
    pa.B = B;
    pa.V = V;
    vt::plan_probs(B, V, h->num_sms, &pa.splits, &pa.range);
    if ((size_t)B * pa.splits > h->probs_part_cap)
      return set_err(h, VT_ERR_CAPACITY, "probability partials exceed their buffer");
    pa.vec_in = ((uintptr_t)logits % 16 == 0) && (((uint64_t)ld * es) % 16 == 0);
    pa.vec_out = ((uintptr_t)out_probs % 16 == 0) && (((uint64_t)ld_probs * 4) % 16 == 0);
    pa.params = h->d_params;
    const bool has_counts = h->counts_B > 0 && h->cfg.max_history > 0;
    pa.hist = has_counts ? h->d_hist : nullptr;
    pa.hist_len = h->d_hist_len;
    pa.hist_cap = h->cfg.max_history > 0 ? h->cfg.max_history : 1;
    pa.tokens = out_tokens;
    pa.row_status = h->d_status;
    pa.kth_value = h->d_kth_v;
    pa.kth_index = h->d_kth_i;
    pa.part = h->d_probs_part;
    pa.probs = out_probs;
    pa.ld_probs = ld_probs;
    VT_CK(h, vt::launch_probs(pa, dtype, st));
    h->last_launches += 2;
    if (update_counts) {
      VT_CK(h, vt::launch_append(h->d_hist, h->d_hist_len, pa.hist_cap, out_tokens, h->d_status,
                                 B, st));
      h->last_launches += 1;
    }
  }
  h->last_B = B;
  h->last_stream = st;
  h->err.clear();
  return VT_OK;
}

int vt_sample(vt_sampler* h, const void* logits, int32_t dtype, int32_t B, int32_t V, int64_t ld,
              int32_t num_logprobs, int32_t update_counts, int32_t* out_tokens,
              float* out_logprobs, int32_t* out_topk_ids, float* out_topk_logprobs,
              void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return set_err(h, VT_ERR_CUDA, "cannot select device %d", h->cfg.device);
  return sample_impl(h, logits, dtype, B, V, ld, num_logprobs, update_counts, out_tokens,
                     out_logprobs, out_topk_ids, out_topk_logprobs, nullptr, 0,
                     (cudaStream_t)stream);
}

int vt_sample_ex(vt_sampler* h, const void* logits, int32_t dtype, int32_t B, int32_t V,
                 int64_t ld, int32_t num_logprobs, int32_t update_counts, int32_t* out_tokens,
                 float* out_logprobs, int32_t* out_topk_ids, float* out_topk_logprobs,
                 float* out_probs, int64_t ld_probs, void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return set_err(h, VT_ERR_CUDA, "cannot select device %d", h->cfg.device);
  return sample_impl(h, logits, dtype, B, V, ld, num_logprobs, update_counts, out_tokens,
                     out_logprobs, out_topk_ids, out_topk_logprobs, out_probs, ld_probs,
                     (cudaStream_t)stream);
}

int vt_check_device_errors(vt_sampler* h) {
  if (!h) return VT_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  VT_CK(h, cudaStreamSynchronize(h->last_stream));
  VT_CK(h, cudaMemcpy(h->h_err, h->d_err, sizeof(int32_t), cudaMemcpyDeviceToHost));
  const int e = *h->h_err;
  if (e != 0) {
    VT_CK(h, cudaMemset(h->d_err, 0, sizeof(int32_t)));
    if (e & vt::kErrTimeout) return set_err(h, VT_ERR_TIMEOUT, "a device wait ran out");
    return set_err(h, VT_ERR_CUDA, "device error word 0x%x", e);
  }
  return VT_OK;
}

int vt_sample_host_async(vt_sampler* h, const void* host_logits, int32_t dtype, int32_t B,
                         int32_t V, int64_t ld, int32_t n, int32_t update_counts,
                         int32_t* host_tokens, float* host_logprobs, int32_t* host_topk_ids,
                         float* host_topk_logprobs, void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  if (!h->io_copy) return set_err(h, VT_ERR_STATE, "handle created without host_io");
  if (!host_logits || !host_tokens) return set_err(h, VT_ERR_INVALID_ARG, "null host buffer");
  if (n > 0 && (!host_topk_ids || !host_topk_logprobs))
    return set_err(h, VT_ERR_INVALID_ARG, "top-k log-prob outputs are null");
  if (dtype != VT_DTYPE_F32 && dtype != VT_DTYPE_BF16)
    return set_err(h, VT_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  const int es = dtype == VT_DTYPE_F32 ? 4 : 2;
  if (B < 1 || ld < 1) return set_err(h, VT_ERR_INVALID_ARG, "bad shape");
  const size_t bytes = (size_t)B * (size_t)ld * es;
  if (bytes > h->io_bytes) return set_err(h, VT_ERR_CAPACITY, "logits exceed host_io staging");
  DeviceGuard guard(h->cfg.device);
  cudaStream_t st = (cudaStream_t)stream;
  vt_sampler::IoSlot& slot = h->io[h->io_next];
  // the copy-in waits, on the device, for the slot's previous step to finish
  // with its buffers; the step waits for its copy-in
  if (slot.busy) VT_CK(h, cudaStreamWaitEvent(h->io_copy, slot.done, 0));
  VT_CK(h, cudaMemcpyAsync(slot.logits, host_logits, bytes, cudaMemcpyHostToDevice, h->io_copy));
  VT_CK(h, cudaEventRecord(slot.copied, h->io_copy));
  VT_CK(h, cudaStreamWaitEvent(st, slot.copied, 0));
  const int rc = sample_impl(h, slot.logits, dtype, B, V, ld, n, update_counts, slot.tokens,
                             slot.lp, n ? slot.tid : nullptr, n ? slot.tlp : nullptr, nullptr, 0,
                             st);
  if (rc != VT_OK) return rc;
  VT_CK(h, cudaMemcpyAsync(host_tokens, slot.tokens, (size_t)B * 4, cudaMemcpyDeviceToHost, st));
  if (host_logprobs)
    VT_CK(h, cudaMemcpyAsync(host_logprobs, slot.lp, (size_t)B * 4, cudaMemcpyDeviceToHost, st));
  if (n > 0) {
    VT_CK(h, cudaMemcpyAsync(host_topk_ids, slot.tid, (size_t)B * n * 4, cudaMemcpyDeviceToHost,
                             st));
    VT_CK(h, cudaMemcpyAsync(host_topk_logprobs, slot.tlp, (size_t)B * n * 4,
                             cudaMemcpyDeviceToHost, st));
  }
  VT_CK(h, cudaEventRecord(slot.done, st));
  slot.busy = true;
  h->io_next ^= 1;
  return VT_OK;
}

int vt_sample_host_wait(vt_sampler* h) {
  if (!h) return VT_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  for (auto& slot : h->io) {
    if (!slot.busy) continue;
    slot.busy = false;
    VT_CK(h, cudaEventSynchronize(slot.done));
  }
  return vt_check_device_errors(h);
}

int vt_sample_host(vt_sampler* h, const void* host_logits, int32_t dtype, int32_t B, int32_t V,
                   int64_t ld, int32_t n, int32_t update_counts, int32_t* host_tokens,
                   float* host_logprobs, int32_t* host_topk_ids, float* host_topk_logprobs,
                   void* stream) {
  const int rc = vt_sample_host_async(h, host_logits, dtype, B, V, ld, n, update_counts,
                                      host_tokens, host_logprobs, host_topk_ids,
                                      host_topk_logprobs, stream);
  if (rc != VT_OK) return rc;
  return vt_sample_host_wait(h);
}

int vt_get_row_status(vt_sampler* h, int32_t* dev_status, void* stream) {
  if (!h || !dev_status) return VT_ERR_INVALID_ARG;
  if (h->last_B == 0) return set_err(h, VT_ERR_STATE, "no vt_sample yet");
  DeviceGuard guard(h->cfg.device);
  VT_CK(h, cudaMemcpyAsync(dev_status, h->d_status, (size_t)h->last_B * 4,
                           cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
  return VT_OK;
}

int vt_debug_filter_boundary(vt_sampler* h, float* kth_value, int32_t* kth_index,
                             int32_t* kept_count, void* stream) {
  if (!h || !kth_value || !kth_index || !kept_count) return VT_ERR_INVALID_ARG;
  if (h->last_B == 0) return set_err(h, VT_ERR_STATE, "no vt_sample yet");
  DeviceGuard guard(h->cfg.device);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t b = (size_t)h->last_B * 4;
  VT_CK(h, cudaMemcpyAsync(kth_value, h->d_kth_v, b, cudaMemcpyDeviceToDevice, st));
  VT_CK(h, cudaMemcpyAsync(kth_index, h->d_kth_i, b, cudaMemcpyDeviceToDevice, st));
  VT_CK(h, cudaMemcpyAsync(kept_count, h->d_kept, b, cudaMemcpyDeviceToDevice, st));
  return VT_OK;
}

int vt_debug_get_counts(vt_sampler* h, int32_t row, int32_t* ids, int32_t* counts,
                        int32_t capacity, int32_t* n_unique) {
  if (!h || !n_unique || capacity < 0 || (capacity > 0 && (!ids || !counts)))
    return VT_ERR_INVALID_ARG;
  if (row < 0 || row >= h->cfg.max_batch) return set_err(h, VT_ERR_INVALID_ARG, "bad row");
  DeviceGuard guard(h->cfg.device);
  VT_CK(h, cudaStreamSynchronize(h->last_stream));
  int32_t len = 0;
  VT_CK(h, cudaMemcpy(&len, h->d_hist_len + row, 4, cudaMemcpyDeviceToHost));
  *n_unique = len;
  const int m = len < capacity ? len : capacity;
  if (m > 0) {
    const int cap = h->cfg.max_history > 0 ? h->cfg.max_history : 1;
    std::vector<int2> tmp(m);
    VT_CK(h, cudaMemcpy(tmp.data(), h->d_hist + (size_t)row * cap, (size_t)m * sizeof(int2),
                        cudaMemcpyDeviceToHost));
    for (int i = 0; i < m; ++i) {
      ids[i] = tmp[i].x;
      counts[i] = tmp[i].y;
    }
  }
  return VT_OK;
}

int vt_debug_set_trace(vt_sampler* h, uint64_t* dev_trace, int64_t capacity_ctas,
                       int32_t* slots_per_cta) {
  if (!h || capacity_ctas < 0 || (capacity_ctas > 0 && !dev_trace)) return VT_ERR_INVALID_ARG;
  h->trace = reinterpret_cast<unsigned long long*>(dev_trace);
  h->trace_ctas = dev_trace ? capacity_ctas : 0;
  if (slots_per_cta) *slots_per_cta = vt::kTraceSlots;
  return VT_OK;
}

int vt_debug_last_handover(vt_sampler* h, int32_t* rows) {
  if (!h || !rows) return VT_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  VT_CK(h, cudaStreamSynchronize(h->last_stream));
  uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  VT_CK(h, cudaMemcpy(v, h->d_slow_ctl, sizeof v, cudaMemcpyDeviceToHost));
  *rows = (int32_t)(v[2] + (h->last_pairs > 1 ? v[6] : 0u));
  return VT_OK;
}

// ---- the vocabulary-sharded sampler ------------------------------------------
int64_t vt_shard_part_bytes(int32_t K) {
  if (K < 1 || K > VT_SHARD_MAX_K) return -1;
  return vt::shard_part_bytes(K);
}

// Rows the sharded path settles exactly: no penalties, no top-p decay, and a
// sampled row's kept set inside a top-k of at most K.
static int shard_rows_ok(vt_sampler* h, int32_t B, int32_t V, int32_t K) {
  if (h->params_B == 0) return set_err(h, VT_ERR_STATE, "sharded call before vt_reset_params");
  if (B < 1 || B > h->params_B)
    return set_err(h, B < 1 ? VT_ERR_INVALID_ARG : VT_ERR_STATE,
                   "B=%d but parameters were reset for %d rows", B, h->params_B);
  if (V < 1 || V > (1 << 20)) return set_err(h, VT_ERR_INVALID_ARG, "V=%d out of range", V);
  if (K < 1 || K > VT_SHARD_MAX_K) return set_err(h, VT_ERR_INVALID_ARG, "K=%d out of range", K);
  for (int r = 0; r < B; ++r) {
    const uint32_t f = h->row_flags[r];
    if (f & (vt::kRowPenalty | vt::kRowDecay))
      return set_err(h, VT_ERR_INVALID_ARG, "row %d: penalties or top-p decay are not sharded", r);
    if (f & vt::kRowGreedy) continue;
    const int k = h->h_params[r].top_k;
    const bool topk = k > 1 && k < V;
    if (!topk && !(f & (vt::kRowTopP | vt::kRowMinP))) continue;  // no filter: every element kept
    if (!(topk && k <= K))
      return set_err(h, VT_ERR_INVALID_ARG,
                     "row %d: a filtered row needs 1 < top_k <= K (%d) and top_k < V (top_k=%d)",
                     r, K, k);
  }
  return VT_OK;
}

int vt_shard_partials(vt_sampler* h, const void* logits, int32_t dtype, int32_t B, int32_t Vs,
                      int64_t ld, int32_t v0, int32_t V, int32_t K, void* part, void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  const int rc = shard_rows_ok(h, B, V, K);
  if (rc != VT_OK) return rc;
  if (dtype != VT_DTYPE_F32 && dtype != VT_DTYPE_BF16)
    return set_err(h, VT_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (!logits || !part) return set_err(h, VT_ERR_INVALID_ARG, "null logits or partials");
  if (Vs < 1 || ld < Vs || v0 < 0 || (int64_t)v0 + Vs > V)
    return set_err(h, VT_ERR_INVALID_ARG, "need 1 <= Vs <= ld and 0 <= v0, v0 + Vs <= V");
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return set_err(h, VT_ERR_CUDA, "cannot select device %d", h->cfg.device);
  vt::ShardArgs a;
  std::memset(&a, 0, sizeof a);
  a.logits = logits;
  a.ld = ld;
  a.B = B;
  a.Vs = Vs;
  a.v0 = v0;
  a.V = V;
  a.K = K;
  a.params = h->d_params;
  a.seeds = h->d_seeds;
  a.part = part;
  a.part_bytes = vt::shard_part_bytes(K);
  cudaStream_t st = (cudaStream_t)stream;
  VT_CK(h, vt::launch_shard_partials(a, dtype, st));
  h->last_stream = st;
  h->err.clear();
  return VT_OK;
}

int vt_shard_merge(vt_sampler* h, const void* parts, int32_t S, int32_t B, int32_t V, int32_t K,
                   int32_t num_logprobs, int32_t* out_tokens, float* out_logprobs,
                   int32_t* out_topk_ids, float* out_topk_logprobs, void* stream) {
  if (!h) return VT_ERR_INVALID_ARG;
  const int rc = shard_rows_ok(h, B, V, K);
  if (rc != VT_OK) return rc;
  if (S < 1 || S > 64 || S * K > VT_SHARD_MAX_RECORDS)
    return set_err(h, VT_ERR_INVALID_ARG, "S=%d: need 1 <= S <= 64 and S * K <= %d", S,
                   VT_SHARD_MAX_RECORDS);
  if (num_logprobs < 0 || num_logprobs > h->cfg.max_logprobs || num_logprobs > K)
    return set_err(h, VT_ERR_INVALID_ARG, "num_logprobs=%d outside [0, min(max_logprobs, K)]",
                   num_logprobs);
  if (!parts || !out_tokens) return set_err(h, VT_ERR_INVALID_ARG, "null partials or tokens");
  if (num_logprobs > 0 && (!out_topk_ids || !out_topk_logprobs))
    return set_err(h, VT_ERR_INVALID_ARG, "top-n log-prob outputs are null");
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return set_err(h, VT_ERR_CUDA, "cannot select device %d", h->cfg.device);
  vt::ShardArgs a;
  std::memset(&a, 0, sizeof a);
  a.B = B;
  a.V = V;
  a.K = K;
  a.S = S;
  a.n_logprobs = num_logprobs;
  a.params = h->d_params;
  a.seeds = h->d_seeds;
  a.part = const_cast<void*>(parts);
  a.part_bytes = vt::shard_part_bytes(K);
  a.out_tokens = out_tokens;
  a.out_logprobs = out_logprobs;
  a.out_topk_ids = out_topk_ids;
  a.out_topk_logprobs = out_topk_logprobs;
  a.row_status = h->d_status;
  a.dbg_kth_value = h->d_kth_v;
  a.dbg_kth_index = h->d_kth_i;
  a.dbg_kept = h->d_kept;
  a.err_word = h->d_err;
  cudaStream_t st = (cudaStream_t)stream;
  VT_CK(h, vt::launch_shard_merge(a, st));
  h->last_B = B;
  h->last_stream = st;
  h->err.clear();
  return VT_OK;
}

int vt_debug_wait_probe(vt_sampler* h, int64_t limit_ns, void* stream) {
  if (!h || limit_ns < 1 || limit_ns > 1000000000LL) return VT_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  cudaStream_t st = (cudaStream_t)stream;
  VT_CK(h, vt::launch_wait_probe(h->d_err, (unsigned long long)limit_ns, st));
  h->last_stream = st;
  return VT_OK;
}

int vt_debug_set_path(vt_sampler* h, int32_t path) {
  if (!h || path < 1 || path > 2) return VT_ERR_INVALID_ARG;
  h->path = path;
  return VT_OK;
}

int vt_debug_last_launches(vt_sampler* h, int32_t* launches) {
  if (!h || !launches) return VT_ERR_INVALID_ARG;
  *launches = h->last_launches;
  return VT_OK;
}

int vt_debug_set_phase_event(vt_sampler* h, void* event) {
  if (!h) return VT_ERR_INVALID_ARG;
  h->phase_event = static_cast<cudaEvent_t>(event);
  return VT_OK;
}

int vt_debug_launch_shape(vt_sampler* h, int32_t dtype, int32_t V, int32_t* ctas_per_row,
                          int32_t* slice_elems, int64_t* smem_bytes) {
  if (!h || !ctas_per_row || (dtype != VT_DTYPE_F32 && dtype != VT_DTYPE_BF16) || V < 1)
    return VT_ERR_INVALID_ARG;
  const int B = h->params_B > 0 ? h->params_B : h->cfg.max_batch;
  DeviceGuard guard(h->cfg.device);
  const vt::LaunchPlan p =
      vt::plan_sample(B, V, dtype == VT_DTYPE_F32 ? 4 : 2, false, dtype, h->num_sms);
  *ctas_per_row = p.cluster;
  if (slice_elems) *slice_elems = p.slice;
  if (smem_bytes) *smem_bytes = (int64_t)p.smem;
  return VT_OK;
}

int vt_debug_get_seeds(vt_sampler* h, uint64_t* host_seeds) {
  if (!h || !host_seeds) return VT_ERR_INVALID_ARG;
  if (h->params_B == 0) return set_err(h, VT_ERR_STATE, "no vt_reset_params yet");
  DeviceGuard guard(h->cfg.device);
  VT_CK(h, cudaStreamSynchronize(h->last_stream));
  VT_CK(h, cudaMemcpy(host_seeds, h->d_seeds, (size_t)h->params_B * 8, cudaMemcpyDeviceToHost));
  return VT_OK;
}

int vt_debug_probs_plan(int32_t B, int32_t V, int32_t num_sms, int32_t* splits, int32_t* range) {
  if (B < 1 || V < 1 || num_sms < 1 || !splits || !range) return VT_ERR_INVALID_ARG;
  vt::plan_probs(B, V, num_sms, splits, range);
  return VT_OK;
}

int vt_read_top_p(vt_sampler* h, float* host_top_p) {
  if (!h || !host_top_p) return VT_ERR_INVALID_ARG;
  if (h->params_B == 0) return set_err(h, VT_ERR_STATE, "no vt_reset_params yet");
  DeviceGuard guard(h->cfg.device);
  VT_CK(h, cudaStreamSynchronize(h->last_stream));
  VT_CK(h, cudaMemcpy(h->h_decay, h->d_decay, (size_t)h->params_B * sizeof(vt::DecayState),
                      cudaMemcpyDeviceToHost));
  for (int r = 0; r < h->params_B; ++r) host_top_p[r] = h->h_decay[r].p;
  return VT_OK;
}

}  // extern "C"
