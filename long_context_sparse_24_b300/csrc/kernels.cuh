// Kernel parameter blocks and launchers shared by the C ABI layer and the kernel files.
#pragma once

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace lcsa {

// Kernel attributes (maximum dynamic shared memory, shared-memory carveout) belong to one device
// context, so every launcher sets them once per device ordinal, under a lock (launchers may be
// called from several host threads).
constexpr int kMaxDevices = 64;
struct PerDeviceOnce {
  std::mutex mu;
  std::atomic<bool> done[kMaxDevices];
};
template <typename F>
cudaError_t once_per_device(PerDeviceOnce& once, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (once.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(once.mu);
  if (once.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess) once.done[dev].store(true, std::memory_order_release);
  return e;
}

struct CompressParams {
  const int32_t* cu_new;
  const int32_t* seq_len;
  int num_seqs;
  const __nv_bfloat16* raw;
  const float* w;
  const float* bias;
  int m;
  int overlap;
  const __nv_bfloat16* pending;
  __nv_bfloat16* pending_out;
  int pending_slots;
  const __nv_bfloat16* scores;         // per-channel weights: score rows of the new tokens, else null
  __nv_bfloat16* pending_scores;       // and of the pending tokens (same ring as pending)
  Rows entries;
  Paging paging;
  Rows new_rows;   // nope == nullptr: write the window ring instead
  Rows window;
  int state_tail;  // > 0: without new_rows, only the last state_tail new tokens reach the state
  int32_t* status;
};

// Per-run top-k lists of the fused decode indexer (workspace): run r of query q keeps up to k
// keys (score key << 32 | ~j) at keys[(q*runs + r)*k ..] and their count at cnt[q*runs + r];
// ticket[b] counts the sequence's finished runs (zero between calls).
struct TopkRuns {
  int runs;
  int* cnt;         // [T][runs] keys in each run's list
  uint64_t* tau;    // [T][runs] the run's selection threshold (0 when it kept every candidate)
  uint64_t* keys;   // [T][runs][list_cap] each run's list, ascending entry index
  int list_cap;     // keys a run's list holds at most (k + k/4, k + k/8, or k: exact lists)
  int* ticket;
  uint64_t* gthr;   // [T] the query's threshold shared by its runs (zero between calls), or null
};

// A run's list: its keys at or above a threshold with k to k + k/4 keys at or above it (all of
// them when it has fewer than k), so that its selection may stop at a digit bin that leaves a few
// more than k; or exactly its k largest (list capacity k).
__host__ __device__ constexpr int topk_list_cap(int k) { return k + (k >> 2); }

struct IndexParams {
  const int32_t* cu_new;
  const int32_t* seq_len;
  int num_seqs;
  const uint8_t* q_fp4;     // [T][Hi][r/2]
  const uint8_t* q_scale;   // [T][Hi][r/32]
  const float* head_w;      // [T][Hi] or null
  int heads;
  const uint8_t* k_fp4;     // [rows][r/2]
  const uint8_t* k_scale;   // [rows][r/32]
  long long k_rows;
  Paging paging;
  int m;
  int relu;
  uint32_t* keys_out;       // [T][ld] order-preserving keys, or
  float* scores_out;        // [T][ld] fp32 scores
  uint32_t* hist;           // [T][2048] histogram of key >> 21 (with keys_out), zeroed by the caller
  long long ld;
  // fused top-k (tensor-core decode scorer)
  int top_k;
  int cand_cap;             // candidate buffer per query (2k + 256)
  int merge_inline;         // 1: the sequence's last CTA merges the run lists
  TopkRuns runs;
  int32_t* out_idx;         // [T][k]
  int32_t* out_cnt;         // [T]
  uint32_t wait_polls;      // bound of every mbarrier wait (polls of up to ~1 us)
  int32_t* status;
};

struct AttendParams {
  const int32_t* cu_new;
  const int32_t* seq_len;
  int num_seqs;
  const __nv_bfloat16* q;
  int heads;
  const int32_t* topk_idx;   // CSA; null -> HCA
  const int32_t* topk_cnt;
  int k;
  int m;
  Rows entries;
  Paging paging;
  Rows window;
  Rows new_rows;
  int sv;                    // 1: separate value rows (warp-MMA kernel only)
  Rows v_entries;            // value rows numbered like entries / window / new_rows
  Rows v_window;
  Rows v_new_rows;
  float scale_log2;
  const float* sink;         // [heads] sink logits folded into the softmax (natural log), or null
  __nv_bfloat16* out;
  float* out_lse;
  float* ws_o;               // [T][H][splits][D] fp32 partials (warp-MMA kernel), or
  __nv_bfloat16* ws_ob;      // [T][H][splits][D] BF16 partials (tensor-core kernel)
  float* ws_ml;              // [T][H][splits][2]
  int splits;
  int rows_per_split;
  int tc;                    // 1: tensor-core kernel (128-row tiles, rows_per_split == 128)
  int entry_splits;          // tensor-core kernel: splits over the entries; split entry_splits = window
  int part;                  // tensor-core kernel: 0 every split, 1 the window split only, 2 the entry splits
  int window_split;          // tensor-core kernel: 1 the window rows form split entry_splits (CSA)
  uint32_t wait_polls;       // bound of every mbarrier wait (polls of up to ~1 us)
  int32_t* status;
};

cudaError_t launch_compress(const CompressParams& p, int D, int max_new, cudaStream_t st);
cudaError_t launch_window_commit(const int32_t* cu_new, const int32_t* seq_len, int num_seqs, int max_new,
                                 const Rows& src, const Rows& ring, int32_t* status, cudaStream_t st);
cudaError_t launch_index_scores(const IndexParams& p, int rank, int max_new, int max_entries, cudaStream_t st);
constexpr int kTopkHistBins = 2048;   // bins of the per-query score-key histogram (key >> 21)
cudaError_t launch_topk_select(const uint32_t* keys, const uint32_t* hist, long long ld, const int32_t* cu_new,
                               const int32_t* seq_len, int num_seqs, int max_new, int m, int k, int32_t* out_idx,
                               int32_t* out_cnt, cudaStream_t st);
// tcgen05 scorer for a few queries per sequence: query-head columns it would use (0 = not applicable)
struct IndexTcPlan {
  int applies;        // 0: the scorer (with k > 0: the fused top-k) does not take this batch
  int qh;             // query-head columns per 32-code block
  int groups;         // query groups per sequence (qh / heads queries each)
  int runs;           // CTAs per query group
  int tpc;            // 128-entry tiles per CTA
  int cap;            // candidate buffer per query (fused)
  int stages;         // shared-memory ring depth
  int list_cap;       // keys of a run's list: topk_list_cap(k), else k + k/8, when the lists then
                      // still fit the last CTA's staging room, else k (exact per-run selection)
  int merge_inline;   // the sequence's last CTA merges (else the merge kernel)
  size_t smem;        // dynamic shared memory of the scorer
  size_t merge_smem;  // dynamic shared memory of the merge kernel
};
// k > 0: plan of the fused top-k; k = 0: of the scores (csa_index_scores)
IndexTcPlan plan_index_tc(const IndexParams& p, int rank, int max_new, int max_entries, int num_seqs, int sms, int k);
cudaError_t launch_index_tc(const IndexParams& p, const IndexTcPlan& plan, cudaStream_t st);
cudaError_t launch_topk_merge(const IndexParams& p, const IndexTcPlan& plan, int max_new, cudaStream_t st);
// tcgen05 scorer for long runs of queries per sequence (prefill chunks)
bool index_tc_pf_applies(const IndexParams& p, int rank, int max_new);
cudaError_t launch_index_tc_pf(const IndexParams& p, int rank, int max_new, int max_entries, cudaStream_t st);
cudaError_t launch_attend(const AttendParams& p, int D, int fmt, int total_new, cudaStream_t st);
cudaError_t launch_attend_tc(const AttendParams& p, int total_new, cudaStream_t st);
cudaError_t launch_attend_tc1(const AttendParams& p, int total_new, cudaStream_t st);
cudaError_t launch_attend_combine(const AttendParams& p, int total_new, int D, cudaStream_t st);
// rows of one query the tensor-core attention takes at most (per 64-head group)
constexpr int kAttendTcMaxRows = 2048 + 128;

}  // namespace lcsa
