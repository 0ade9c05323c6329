// vt_kernels.h -- internal interface between the C-ABI host code and the
// CUDA kernels of the sampler (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vt {

struct RowParams;
struct DecayState;

// A row the streaming kernel hands to the selection kernel.
struct __align__(16) SlowRow {
  float m_t;      // tempered row maximum
  float lnS;      // ln(sum exp(z_t - m_t))
  float xmax;     // row maximum before temperature
  uint32_t bi_topn;  // lowest index of the maximum; bit 31: top-n outputs already written
};

// Everything one sampling launch needs.  Device pointers unless noted.
struct SampleArgs {
  const void* logits;        // [rows][ld] elements
  int64_t ld;                // row stride in elements
  int32_t B, V;              // B: rows of this launch (the grid is B * cluster CTAs)
  const int32_t* rows;       // [B] the rows of this launch, or null for rows 0..B-1
  int32_t early;             // hand every row over after its statistics
  int32_t n_logprobs;
  int32_t update_counts;
  int32_t slice;             // elements per CTA (multiple of 32)
  int32_t aligned;           // rows 16-byte aligned: 16-byte vector loads
  int32_t pen_smem;          // dynamic smem holds the penalty bitmap and prefix
  uint32_t off_gmax;         // dynamic smem offsets (bytes)
  uint32_t off_mrg;
  uint32_t off_bitmap;
  uint32_t off_prefix;
  const RowParams* params;   // [B]
  uint64_t* seeds;           // [B], advanced by the kernel
  DecayState* decay;         // [B] top-p decay state (rows with kRowDecay), may be null
  int2* hist;                // [B][hist_cap] sorted (id, count)
  int32_t* hist_len;         // [B]
  int32_t hist_cap;
  float* zside;              // [B][hist_cap] penalised logits of the table entries
  int32_t* out_tokens;
  float* out_logprobs;       // may be null
  int32_t* out_topk_ids;     // [B][n], may be null when n == 0
  float* out_topk_logprobs;
  int32_t* row_status;       // [B]
  float* dbg_kth_value;      // [B]
  int32_t* dbg_kth_index;    // [B]
  int32_t* dbg_kept;         // [B]
  int32_t* err_word;         // one int, kErr* bits
  SlowRow* slow;             // [B] hand-over records
  int32_t* slow_list;        // [B] rows handed over, in arrival order
  uint32_t* slow_ctl;        // [3] rows handed over, selection CTAs done (both zero between
                             // calls), rows handed over by the last call
  unsigned long long* trace; // optional [grid][kTraceSlots] phase timestamps (ns)
  int64_t trace_ctas;        // CTAs the trace buffer holds
};

// Launch shape of the selection kernel (kernel 2).
struct SelectPlan {
  int cluster;          // CTAs per row
  int slice;            // elements per CTA
  int pen_smem;
  int staged;           // the slice is copied into shared memory
  uint32_t off_gmax, off_mrg, off_bitmap, off_prefix, off_stage;
  uint32_t off_code;     // bf16 code-slot histograms (0: none)
  size_t smem;
  int clusters;         // persistent clusters launched
  int kernel1_cluster;  // CTAs per row of the streaming kernel (trace layout)
};

constexpr int kTraceSlots = 16;

struct LaunchPlan {
  int cluster;        // CTAs per row
  int slice;          // elements per CTA
  int pen_smem;       // penalty bitmap in shared memory
  uint32_t off_gmax, off_mrg, off_bitmap, off_prefix;
  size_t smem;        // dynamic shared memory per CTA
  int active_clusters;  // clusters resident at once (filled by prepare_sample)
  SelectPlan sel;       // the selection kernel that finishes handed-over rows
  SelectPlan own;       // the selection kernel taking its rows' statistics itself
                        // (bf16 only; cluster 0 otherwise)
};

// Shared-memory layout for V elements of elem_size bytes split over `cluster`
// CTAs (1, 2, 4, 8 or 16), for the streaming kernel (select = false) or the
// selection kernel (select = true, without its staged slice).
LaunchPlan plan_layout(int V, int elem_size, int cluster, bool penalties, bool select);

// Choose the cluster size for a call: as many CTAs per row as still lets all
// B rows be resident in one wave, within the slice-size limits.
LaunchPlan plan_sample(int B, int V, int elem_size, bool penalties, int dtype, int num_sms);

// Prepare kernel attributes (dynamic smem, non-portable clusters); fills
// plan.active_clusters.  Returns a cudaError_t.
cudaError_t prepare_sample(LaunchPlan& plan, int dtype);

// Launch the sampling kernels: the streaming kernel (grid B * cluster CTAs),
// then the selection kernel for the rows it handed over.
cudaError_t launch_sample(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                          cudaStream_t stream, cudaEvent_t between = nullptr);

// The selection kernel alone over the rows args.rows[0, args.B) (args.early
// set): one cluster per row streams its slices for the row statistics (the
// same slices and arithmetic as the streaming kernel), then selects and draws.
// `launched`, when not null, is recorded once every CTA of the launch has begun.
cudaError_t launch_select_own(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                              cudaStream_t stream, cudaEvent_t launched = nullptr);

// One CTA of one thread waits, at most limit_ns, on a barrier nothing
// completes, then sets kErrTimeout in *err_word (the bounded-wait path of the
// sampling kernels, made to run out).
cudaError_t launch_wait_probe(int32_t* err_word, unsigned long long limit_ns,
                              cudaStream_t stream);

// Build the per-row sorted (id, count) tables from raw ids.
//   raw, offs  CSR: row r owns raw[offs[r] .. offs[r+1]) (prompt then output)
//   max_len    the longest row (sizes the shared-memory sort)
//   hist       [B][hist_cap] output, hist_len[B] output
cudaError_t launch_build_counts(const int32_t* raw, const int64_t* offs, int max_len, int B,
                                int2* hist, int32_t* hist_len, int32_t hist_cap,
                                cudaStream_t stream);

// Append each sampled row's token to its count table (rows whose status is
// not ok are left alone; a full table sets status VT_ROW_HISTORY_FULL), as
// the sampling kernels do when they update the counts themselves.
cudaError_t launch_append(int2* hist, int32_t* hist_len, int32_t hist_cap, const int32_t* tokens,
                          int32_t* row_status, int B, cudaStream_t stream);

// ---- the flat kernels (vt_flat.cu) -------------------------------------------
// bf16 batches without penalties or top-p decay, rows 16-byte aligned.  Six
// launches, none of whose CTAs waits on another: per-slice statistics (one
// read of the logits from HBM), per-row statistics and thresholds, per-slice
// collection (candidates, code-slot mass histograms, draw contenders; a second
// read, from L2), per-row completion of the rows the candidates settle, and for
// top-p rows a fine count inside the boundary bin and the row's completion.
// Rows none of them settles exactly go to the selection kernel through the
// SlowRow records.
constexpr int kFlatMaxC = 32;        // slices per row at most
constexpr int kFlatMaxNV = 12;       // 16-byte vectors per thread of a slice
constexpr int kFlatCandCap = 4096;   // candidate keys per row
constexpr int kFlatContCap = 512;    // draw contenders per row
constexpr int kFlatKMax = 1024;      // largest top_k the candidates settle
constexpr int kFlatBins = 64;        // coarse bins of 64 code slots

struct FlatPlan {
  int C;   // slices per row (0: the flat kernels do not take this width)
  int L;   // elements per slice, a multiple of 8
  int NV;  // 16-byte vectors per thread
};

struct FlatArgs {
  const void* logits;  // [B][ld] bf16
  int64_t ld;
  int32_t B, V, C, L, NV;
  int32_t n_logprobs;
  const RowParams* params;
  uint64_t* seeds;
  int32_t* out_tokens;
  float* out_logprobs;       // may be null
  int32_t* out_topk_ids;     // [B][n]
  float* out_topk_logprobs;
  int32_t* row_status;
  float* dbg_kth_value;
  int32_t* dbg_kth_index;
  int32_t* dbg_kept;
  SlowRow* slow;             // hand-over records and list, as SampleArgs
  int32_t* slow_list;
  uint32_t* slow_ctl;
  void* scratch;             // flat_scratch_bytes(B, C) bytes
};

FlatPlan plan_flat(int V);
size_t flat_scratch_bytes(int B, int C);
// The six launches on `stream`; the caller then launches the selection kernel
// for the rows handed over (launch_select_handed).
cudaError_t launch_flat(const FlatArgs& a, cudaStream_t stream);

// The selection kernel alone over the rows another launch handed over
// (max_clusters > 0: at most that many of its clusters).
cudaError_t launch_select_handed(const SampleArgs& args, const LaunchPlan& plan, int dtype,
                                 cudaStream_t stream,
                                 int max_clusters = 0);

// ---- the vocabulary-sharded sampler (vt_shard.cu) ---------------------------
struct ShardArgs {
  const void* logits;        // partials: the shard's columns [B][ld]
  int64_t ld;
  int32_t B, Vs, v0, V;      // rows, shard width, its first global column, the row width
  int32_t K;                 // records per row and shard (<= 256)
  int32_t S;                 // merge: shards
  int32_t n_logprobs;
  const RowParams* params;   // [B]
  uint64_t* seeds;           // [B], advanced by the merge
  void* part;                // partials: [B] records; merge: [S][B] records
  int64_t part_bytes;        // bytes of one row's record
  int32_t* out_tokens;
  float* out_logprobs;
  int32_t* out_topk_ids;
  float* out_topk_logprobs;
  int32_t* row_status;
  float* dbg_kth_value;
  int32_t* dbg_kth_index;
  int32_t* dbg_kept;
  int32_t* err_word;
};
int64_t shard_part_bytes(int K);
cudaError_t launch_shard_partials(const ShardArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_shard_merge(const ShardArgs& a, cudaStream_t stream);

// ---- the filtered distribution on request (vt_probs.cu) ---------------------
constexpr int kProbsMaxRange = 65536;  // elements per CTA at most
constexpr int kProbsMaxSplits = 64;    // CTAs per row at most (unless V needs more)
constexpr int kProbsCtasPerSm = 6;     // the grid aims at this many CTAs per SM

struct ProbsArgs {
  const void* logits;          // [B][ld] elements, as sampled
  int64_t ld;
  int32_t B, V;
  int32_t splits, range;       // CTAs per row, elements per CTA (multiple of 64)
  int32_t vec_in;              // rows 16-byte aligned: 16-byte loads
  int32_t vec_out;             // output rows 16-byte aligned: 16-byte stores
  const RowParams* params;     // [B]
  const int2* hist;            // [B][hist_cap] sorted (id, count), may be null
  const int32_t* hist_len;
  int32_t hist_cap;
  const int32_t* tokens;       // [B] the drawn tokens
  const int32_t* row_status;   // [B]
  const float* kth_value;      // [B] the last kept element: value, index
  const int32_t* kth_index;
  float2* part;                // [B * splits] (max, exp-sum) partials
  float* probs;                // [B][ld_probs] fp32 output
  int64_t ld_probs;
};

// CTAs per row and elements per CTA for B rows of V.
void plan_probs(int B, int V, int num_sms, int* splits, int* range);

// The two launches (partials, then the probabilities) on `stream`.
cudaError_t launch_probs(const ProbsArgs& args, int dtype, cudaStream_t stream);

}  // namespace vt
