// C ABI entry points: argument validation, workspace layout and kernel launches.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "kernels.cuh"

using namespace lcsa;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lcs_status check_batch(const lcs_batch* b) {
  if (b == nullptr || b->cu_new == nullptr || b->seq_len == nullptr) return LCS_ERR_INVALID_ARG;
  if (b->num_seqs <= 0 || b->num_seqs > 65535) return LCS_ERR_UNSUPPORTED;
  if (b->total_new < 0 || b->max_new < 0 || b->max_seq_len < 0) return LCS_ERR_INVALID_ARG;
  if (b->max_new > b->max_seq_len) return LCS_ERR_SHAPE;
  if ((long long)b->total_new > (long long)b->num_seqs * b->max_new) return LCS_ERR_SHAPE;   // no sequence has more
  return LCS_OK;
}

lcs_status check_rows(const lcs_rows* r, bool need_data = true) {
  if (r == nullptr) return LCS_ERR_INVALID_ARG;
  if (r->dim != 128 && r->dim != 512) return LCS_ERR_UNSUPPORTED;
  if (r->format == LCS_ROW_BF16) {
    if (need_data && r->nope == nullptr) return LCS_ERR_INVALID_ARG;
    if (!aligned16(r->nope)) return LCS_ERR_ALIGNMENT;
  } else if (r->format == LCS_ROW_FP8_SPLIT) {
    if (need_data && (r->nope == nullptr || r->rope == nullptr || r->scale == nullptr)) return LCS_ERR_INVALID_ARG;
    if (!aligned16(r->nope) || !aligned16(r->rope) || (reinterpret_cast<uintptr_t>(r->scale) & 3u))
      return LCS_ERR_ALIGNMENT;
  } else {
    return LCS_ERR_UNSUPPORTED;
  }
  if (r->num_rows < 0) return LCS_ERR_INVALID_ARG;
  return LCS_OK;
}

bool same_layout(const lcs_rows& a, const lcs_rows& b) { return a.format == b.format && a.dim == b.dim; }

lcs_status check_paging(const lcs_paging* p) {
  if (p == nullptr || p->block_table == nullptr) return LCS_ERR_INVALID_ARG;
  if (p->entries_per_block <= 0 || p->max_blocks_per_seq <= 0) return LCS_ERR_INVALID_ARG;
  return LCS_OK;
}

lcs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LCS_OK : LCS_ERR_CUDA; }

int num_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

long long index_ld(const lcs_batch* b, int m) {
  long long n = b->max_seq_len / m;
  return (n + 3) / 4 * 4;
}

struct SplitPlan {
  int splits;
  int rows_per_split;
  int tc;
  int entry_splits;   // tensor-core plan: 128-row tiles of entries; one more split for the window
  int window_apart;   // tensor-core plan: the window rows form their own split (CSA, few queries)
};

// The tensor-core attention takes FP8-split rows of D = 512 (the only D = 512 format), heads in
// groups of 64 (one CTA per group).  CSA with few queries (window_split and less than a wave of
// (query, head group) CTAs): top-k lists up to 2048 entries, one split per 128-row tile of
// entries while a wave has room, plus the window split, so that the window part can run next to
// the indexer.  Otherwise (HCA, or CSA prefill runs that fill the GPU by themselves): one list of
// entries then window rows, cut into about one wave of CTAs.
bool attend_tc_applies(int heads, int dim) { return dim == 512 && heads <= 128; }

SplitPlan plan_splits(const lcs_batch* b, int heads, int dim, int max_rows, bool window_split, bool tc_ok = true) {
  if (tc_ok && attend_tc_applies(heads, dim)) {
    const int sms = num_sms();
    const long long ctas = std::max<long long>(1, (long long)b->total_new * ((heads + 63) / 64));
    const int per_query = (int)std::max<long long>(1, sms / ctas);   // CTAs per (query, head group)
    if (window_split && per_query > 1 && max_rows <= kAttendTcMaxRows) {
      const int tiles = std::max(1, (max_rows - LCSA_WINDOW + 127) / 128);
      const int es = std::min(tiles, per_query);
      const int tps = (tiles + es - 1) / es;
      return SplitPlan{(tiles + tps - 1) / tps + 1, 128 * tps, 1, (tiles + tps - 1) / tps, 1};
    }
    // one list per query: cut it into runs of tps tiles so that all (query, head group) runs
    // together come to about one tile load per SM (the last run of a query may be shorter;
    // CTAs start in split order, so the short runs fill the SMs the long ones leave); with few
    // queries and short lists (CSA top-k plus window in one call), the shortest runs that keep
    // every run in one wave of CTAs
    const int tiles = std::max(1, (max_rows + 127) / 128);
    const long long units = ctas * tiles;
    int tps = (int)std::min<long long>(tiles, std::max<long long>(1, (units + num_sms() - 1) / num_sms()));
    if (ctas * 2 <= sms && tiles <= 32) tps = (tiles + (int)(sms / ctas) - 1) / (int)(sms / ctas);
    const int splits = (tiles + tps - 1) / tps;
    return SplitPlan{splits, 128 * tps, 1, splits, 0};
  }
  const int hg = heads <= 16 ? 1 : (heads + 63) / 64;
  const long long base = (long long)b->total_new * hg;
  SplitPlan s{1, max_rows > 0 ? max_rows : 1, 0, 0, 0};
  const int sms = num_sms();
  if (base <= 0 || base >= sms || max_rows <= 64) return s;
  int want = (int)(sms / base);
  const int cap = (max_rows + 63) / 64;
  if (want > cap) want = cap;
  if (want <= 1) return s;
  int rps = (max_rows + want - 1) / want;
  rps = (rps + 31) / 32 * 32;
  s.rows_per_split = rps;
  s.splits = (max_rows + rps - 1) / rps;
  return s;
}

// Split partials: O [T][H][splits][D] (fp32, or BF16 for the tensor-core kernel), then the
// (max, sum) pairs [T][H][splits][2] fp32.
size_t attend_ws_bytes(const lcs_batch* b, int heads, int dim, const SplitPlan& s) {
  if (s.splits <= 1) return 0;
  const size_t per = (size_t)b->total_new * heads * s.splits;
  return per * dim * (s.tc ? 2 : 4) + per * 2 * 4 + 256;
}

std::atomic<uint32_t> g_wait_polls{LCSA_DEFAULT_WAIT_POLLS};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

constexpr int kFusedMaxQueries = 16;   // queries per sequence up to which the top-k is fused

// Workspace of csa_index_topk.  Both layouts start with the part that is zero between calls: the
// ticket counters (one per sequence and query group, at most int32[num_seqs][max_new]), then the
// queries' shared thresholds (u64[num_seqs][max_new], at least one per batch row).  Fused top-k: run counts
// int32[T][runs], run thresholds u64[T][runs], run keys u64[T][runs][k].  Otherwise: score keys
// u32[T][ld], histograms u32[T][2048].
struct TopkWs {
  bool fused;
  IndexTcPlan plan;
  size_t ticket, gthr, cnt, tau, keys, hist, total;
};

size_t zeroed_tickets_bytes(const lcs_batch* b) {
  return round256((size_t)b->num_seqs * std::max(1, b->max_new) * 4);
}

TopkWs topk_ws_layout(const lcs_batch* b, const IndexParams& p, int rank, int m, int k, int sms) {
  TopkWs w{};
  const size_t T = (size_t)b->total_new;
  w.ticket = 0;
  w.gthr = zeroed_tickets_bytes(b);
  const size_t body = lcs_index_topk_workspace_zeroed(b);
  // the top-k fused into the scorer serves up to 16 queries per sequence (groups of at most 4 per
  // CTA); longer query runs take the prefill scorer, whose CTAs score 16 queries per key tile (a
  // quarter of the key reads) and write every score key for the select kernel
  const bool long_runs = b->max_new > kFusedMaxQueries && index_tc_pf_applies(p, rank, b->max_new);
  if (!long_runs) w.plan = plan_index_tc(p, rank, b->max_new, b->max_seq_len / m, b->num_seqs, sms, k);
  w.fused = w.plan.applies != 0;
  if (w.fused) {
    w.cnt = body;
    w.tau = w.cnt + round256(T * w.plan.runs * 4);
    w.keys = w.tau + round256(T * w.plan.runs * 8);
    w.hist = w.keys;
    w.total = w.keys + T * w.plan.runs * (size_t)w.plan.list_cap * 8 + 256;
  } else {
    w.keys = body;
    w.hist = w.keys + round256(T * (size_t)index_ld(b, m) * 4);
    w.total = w.hist + T * kTopkHistBins * 4 + 256;
  }
  return w;
}

// Indexer scores on their own (csa_index_scores): the tcgen05 scorer for a few queries per
// sequence, the tcgen05 prefill scorer for query runs, the warp-MMA scorer for what neither
// takes (rank 64, other page sizes).
cudaError_t launch_scores(const IndexParams& p, const lcs_batch* b, int rank, int m, cudaStream_t st) {
  const int max_entries = b->max_seq_len / m;
  const IndexTcPlan plan = plan_index_tc(p, rank, b->max_new, max_entries, b->num_seqs, num_sms(), 0);
  if (plan.applies) return launch_index_tc(p, plan, st);
  if (index_tc_pf_applies(p, rank, b->max_new)) return launch_index_tc_pf(p, rank, b->max_new, max_entries, st);
  return launch_index_scores(p, rank, b->max_new, max_entries, st);
}

// Score keys and histograms of every (query, visible entry) for the selection pass: the tcgen05
// prefill scorer for query runs, the warp-MMA scorer otherwise.
cudaError_t launch_score_keys(const IndexParams& p, int rank, int max_new, int max_entries, cudaStream_t st) {
  if (index_tc_pf_applies(p, rank, max_new)) return launch_index_tc_pf(p, rank, max_new, max_entries, st);
  return launch_index_scores(p, rank, max_new, max_entries, st);
}

lcs_status compress_common(const lcs_batch* batch, const void* raw, const lcs_compressor* comp,
                           const lcs_state* state, const lcs_rows* entries, const lcs_paging* paging,
                           int32_t* dev_status, void* stream, bool hca) {
  lcs_status s = check_batch(batch);
  if (s != LCS_OK) return s;
  if (comp == nullptr || state == nullptr || comp->bias == nullptr) return LCS_ERR_INVALID_ARG;
  const bool per_channel = comp->scores != nullptr;
  if (!per_channel && comp->w == nullptr) return LCS_ERR_INVALID_ARG;
  if (raw == nullptr && batch->total_new > 0) return LCS_ERR_INVALID_ARG;
  if (!aligned16(raw) || !aligned16(state->pending)) return LCS_ERR_ALIGNMENT;
  const int m = comp->m;
  if (m <= 0 || m > 128 || (m & (m - 1)) != 0) return LCS_ERR_UNSUPPORTED;
  if (hca && comp->overlap) return LCS_ERR_UNSUPPORTED;
  const int slots = comp->overlap ? 2 * m : m;
  if (state->pending == nullptr || state->pending_slots != slots) return LCS_ERR_SHAPE;
  if (per_channel) {   // the streaming compressor (ratios up to 4) takes per-channel weights
    if (m > 4) return LCS_ERR_UNSUPPORTED;
    if (state->pending_scores == nullptr) return LCS_ERR_INVALID_ARG;
    if (!aligned16(comp->scores) || !aligned16(state->pending_scores)) return LCS_ERR_ALIGNMENT;
  }
  if ((s = check_rows(entries)) != LCS_OK) return s;
  if ((s = check_paging(paging)) != LCS_OK) return s;
  const bool have_new = state->new_rows.nope != nullptr;
  if (have_new) {
    if ((s = check_rows(&state->new_rows)) != LCS_OK) return s;
    if (!same_layout(state->new_rows, *entries)) return LCS_ERR_SHAPE;
    if (state->new_rows.num_rows < batch->total_new) return LCS_ERR_SHAPE;
  } else {
    if ((s = check_rows(&state->window)) != LCS_OK) return s;
    if (!same_layout(state->window, *entries)) return LCS_ERR_SHAPE;
    if (state->window.num_rows < (int64_t)batch->num_seqs * LCSA_WINDOW) return LCS_ERR_SHAPE;
  }
  CompressParams p;
  std::memset(&p, 0, sizeof(p));
  p.cu_new = batch->cu_new;
  p.seq_len = batch->seq_len;
  p.num_seqs = batch->num_seqs;
  p.raw = static_cast<const __nv_bfloat16*>(raw);
  p.w = comp->w;
  p.bias = comp->bias;
  p.m = m;
  p.overlap = comp->overlap ? 1 : 0;
  p.pending = static_cast<const __nv_bfloat16*>(state->pending);
  p.pending_out = static_cast<__nv_bfloat16*>(state->pending);
  p.pending_slots = slots;
  p.scores = static_cast<const __nv_bfloat16*>(comp->scores);
  p.pending_scores = per_channel ? static_cast<__nv_bfloat16*>(state->pending_scores) : nullptr;
  p.entries = make_rows(*entries);
  p.paging = make_paging(*paging);
  p.new_rows = make_rows(state->new_rows);
  if (!have_new) p.new_rows.nope = nullptr;
  p.window = make_rows(state->window);
  // pending rows reach back at most 2m - 1 tokens (overlap) and the ring 128 tokens
  p.state_tail = std::max(LCSA_WINDOW, slots);
  p.status = dev_status;
  return from_cuda(launch_compress(p, entries->dim, batch->max_new, static_cast<cudaStream_t>(stream)));
}

lcs_status index_common(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale, int32_t heads,
                        const lcs_index_keys* keys, const lcs_paging* paging, int32_t m, IndexParams& p) {
  lcs_status s = check_batch(batch);
  if (s != LCS_OK) return s;
  if (q_fp4 == nullptr || q_scale == nullptr || keys == nullptr || keys->fp4 == nullptr || keys->scale == nullptr)
    return LCS_ERR_INVALID_ARG;
  if (heads != 1 && heads != 2 && heads != 4 && heads != 8) return LCS_ERR_UNSUPPORTED;
  if (keys->rank != 64 && keys->rank != 128) return LCS_ERR_UNSUPPORTED;
  if (m <= 0 || m > 128 || (m & (m - 1)) != 0) return LCS_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q_fp4) & 3u) || (reinterpret_cast<uintptr_t>(keys->fp4) & 3u) ||
      (reinterpret_cast<uintptr_t>(keys->scale) & 3u) || (reinterpret_cast<uintptr_t>(q_scale) & 1u))
    return LCS_ERR_ALIGNMENT;
  if ((s = check_paging(paging)) != LCS_OK) return s;
  std::memset(&p, 0, sizeof(p));
  p.cu_new = batch->cu_new;
  p.seq_len = batch->seq_len;
  p.num_seqs = batch->num_seqs;
  p.q_fp4 = q_fp4;
  p.q_scale = q_scale;
  p.heads = heads;
  p.k_fp4 = keys->fp4;
  p.k_scale = keys->scale;
  p.k_rows = keys->num_rows;
  p.paging = make_paging(*paging);
  p.m = m;
  p.wait_polls = g_wait_polls.load(std::memory_order_relaxed);
  return LCS_OK;
}

// Value sets: each one's format, dim and row count equal its key counterpart's (the same row
// numbers address both), and new value rows exist exactly when new key rows do.
lcs_status check_values(const lcs_values* v, const lcs_rows* entries, const lcs_state* state) {
  lcs_status s;
  const lcs_rows* pairs[2][2] = {{&v->entries, entries}, {&v->window, &state->window}};
  for (auto& pr : pairs) {
    if ((s = check_rows(pr[0])) != LCS_OK) return s;
    if (!same_layout(*pr[0], *pr[1]) || pr[0]->num_rows != pr[1]->num_rows) return LCS_ERR_SHAPE;
  }
  if ((v->new_rows.nope != nullptr) != (state->new_rows.nope != nullptr)) return LCS_ERR_SHAPE;
  if (v->new_rows.nope != nullptr) {
    if ((s = check_rows(&v->new_rows)) != LCS_OK) return s;
    if (!same_layout(v->new_rows, state->new_rows) || v->new_rows.num_rows != state->new_rows.num_rows)
      return LCS_ERR_SHAPE;
  }
  return LCS_OK;
}

lcs_status attend_common(const lcs_batch* batch, const void* q, int32_t heads, const lcs_rows* entries,
                         const lcs_paging* paging, const lcs_state* state, const lcs_values* values, void* out,
                         void* workspace, size_t workspace_bytes, int max_rows, AttendParams& p, bool window_split,
                         bool no_out = false) {
  lcs_status s = check_batch(batch);
  if (s != LCS_OK) return s;
  if (q == nullptr || (out == nullptr && !no_out) || state == nullptr) return LCS_ERR_INVALID_ARG;
  if (!(heads == 8 || (heads % 16 == 0 && heads >= 16 && heads <= 128))) return LCS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out)) return LCS_ERR_ALIGNMENT;
  if ((s = check_rows(entries)) != LCS_OK) return s;
  if ((s = check_paging(paging)) != LCS_OK) return s;
  if ((s = check_rows(&state->window)) != LCS_OK) return s;
  if (!same_layout(state->window, *entries)) return LCS_ERR_SHAPE;
  if (state->window.num_rows < (int64_t)batch->num_seqs * LCSA_WINDOW) return LCS_ERR_SHAPE;
  // every query's own token is one of this call's new tokens: its window row comes from new_rows,
  // or, when new_rows is absent, from the ring (one new token per sequence, already in the ring)
  const bool have_new = state->new_rows.nope != nullptr;
  if (have_new) {
    if ((s = check_rows(&state->new_rows)) != LCS_OK) return s;
    if (!same_layout(state->new_rows, *entries)) return LCS_ERR_SHAPE;
    if (state->new_rows.num_rows < batch->total_new) return LCS_ERR_SHAPE;
  } else if (batch->max_new > 1) {
    return LCS_ERR_SHAPE;
  }
  if (entries->num_rows < 1) return LCS_ERR_SHAPE;
  if (entries->format == LCS_ROW_BF16 && entries->dim == 512) return LCS_ERR_UNSUPPORTED;
  if (values != nullptr && (s = check_values(values, entries, state)) != LCS_OK) return s;
  const SplitPlan plan = plan_splits(batch, heads, entries->dim, max_rows, window_split, values == nullptr);
  const size_t need = attend_ws_bytes(batch, heads, entries->dim, plan);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return LCS_ERR_WORKSPACE;
  if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return LCS_ERR_ALIGNMENT;
  std::memset(&p, 0, sizeof(p));
  p.cu_new = batch->cu_new;
  p.seq_len = batch->seq_len;
  p.num_seqs = batch->num_seqs;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.heads = heads;
  p.entries = make_rows(*entries);
  p.paging = make_paging(*paging);
  p.window = make_rows(state->window);
  p.new_rows = make_rows(state->new_rows);
  if (!have_new) {
    p.new_rows.nope = nullptr;
    p.new_rows.num_rows = 0;
  }
  if (values != nullptr) {
    p.sv = 1;
    p.v_entries = make_rows(values->entries);
    p.v_window = make_rows(values->window);
    p.v_new_rows = make_rows(values->new_rows);
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  p.splits = plan.splits;
  p.rows_per_split = plan.rows_per_split;
  p.tc = plan.tc;
  p.entry_splits = plan.entry_splits;
  p.window_split = plan.window_apart;
  p.wait_polls = g_wait_polls.load(std::memory_order_relaxed);
  if (plan.splits > 1) {
    const size_t per = (size_t)batch->total_new * heads * plan.splits;
    const size_t ob = per * entries->dim * (plan.tc ? 2 : 4);
    if (plan.tc) p.ws_ob = static_cast<__nv_bfloat16*>(workspace);
    else p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ob);
  }
  return LCS_OK;
}

lcs_status csa_attend_part(const lcs_batch* batch, const void* q, int32_t heads, const int32_t* topk_idx,
                           const int32_t* topk_cnt, int32_t k, int32_t m, const lcs_rows* entries,
                           const lcs_paging* paging, const lcs_state* state, const lcs_values* values,
                           const float* sink, float softmax_scale, void* out, float* out_lse, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, void* stream, int part) {
  if (topk_idx == nullptr && part != 1) return LCS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 3u) return LCS_ERR_ALIGNMENT;
  if (k < 1 || k > 4096 || m <= 0 || m > 128) return LCS_ERR_UNSUPPORTED;
  AttendParams p;
  // the window rows form a split of their own only for the two-part calls (the window part runs
  // next to the indexer); one call plans the query's entries and window rows as one list
  lcs_status s = attend_common(batch, q, heads, entries, paging, state, values, part == 1 ? nullptr : out,
                               workspace, workspace_bytes, k + LCSA_WINDOW, p, part != 0, part == 1);
  if (s != LCS_OK) return s;
  if (part != 0 && !p.window_split) {
    // only the tensor-core plan for few queries computes the window split apart: otherwise the
    // window call does nothing and the top-k call computes everything
    if (part == 1) return LCS_OK;
    part = 0;
  }
  p.part = part;
  p.topk_idx = topk_idx;
  p.topk_cnt = topk_cnt;
  p.k = k;
  p.m = m;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.sink = part == 1 ? nullptr : sink;
  p.out_lse = out_lse;
  p.status = dev_status;
  return from_cuda(launch_attend(p, entries->dim, entries->format, batch->total_new, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

size_t lcs_index_topk_workspace(const lcs_batch* batch, int32_t heads, const lcs_index_keys* keys,
                                const lcs_paging* paging, int32_t m, int32_t k) {
  if (batch == nullptr || keys == nullptr || paging == nullptr || m <= 0 || k < 1) return 0;
  IndexParams p;
  std::memset(&p, 0, sizeof(p));
  p.heads = heads;
  p.k_fp4 = keys->fp4;
  p.k_scale = keys->scale;
  p.k_rows = keys->num_rows;
  p.paging = make_paging(*paging);
  // (the grid, and so the number of run lists, is largest with every SM: this covers any spare)
  return topk_ws_layout(batch, p, keys->rank, m, k, num_sms()).total;
}

size_t lcs_index_topk_workspace_zeroed(const lcs_batch* batch) {
  if (batch == nullptr) return 0;
  return zeroed_tickets_bytes(batch) + round256((size_t)batch->num_seqs * std::max(1, batch->max_new) * 8);
}

uint32_t lcs_set_wait_polls(uint32_t polls) { return g_wait_polls.exchange(polls); }

int32_t lcs_abi_version(void) { return LCSA_ABI_VERSION; }

const char* lcs_status_string(int32_t s) {
  switch (s) {
    case LCS_OK: return "ok";
    case LCS_ERR_INVALID_ARG: return "invalid argument";
    case LCS_ERR_SHAPE: return "inconsistent shapes";
    case LCS_ERR_ALIGNMENT: return "misaligned buffer";
    case LCS_ERR_UNSUPPORTED: return "unsupported size";
    case LCS_ERR_CUDA: return "CUDA error";
    case LCS_ERR_DEVICE_GUARD: return "device-side index or block id out of range";
    case LCS_ERR_TIMEOUT: return "bounded device wait timed out";
    case LCS_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

lcs_status lcs_device_check(void) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCS_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return LCS_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return LCS_ERR_CUDA;
  return (major == 10 && minor == 3) ? LCS_OK : LCS_ERR_UNSUPPORTED;
}

lcs_status csa_compress(const lcs_batch* batch, const void* raw, const lcs_compressor* comp, const lcs_state* state,
                        const lcs_rows* entries, const lcs_paging* paging, int32_t* dev_status, void* stream) {
  return compress_common(batch, raw, comp, state, entries, paging, dev_status, stream, false);
}

lcs_status hca_compress(const lcs_batch* batch, const void* raw, const lcs_compressor* comp, const lcs_state* state,
                        const lcs_rows* entries, const lcs_paging* paging, int32_t* dev_status, void* stream) {
  return compress_common(batch, raw, comp, state, entries, paging, dev_status, stream, true);
}

lcs_status lcs_window_commit(const lcs_batch* batch, const lcs_state* state, int32_t* dev_status, void* stream) {
  lcs_status s = check_batch(batch);
  if (s != LCS_OK) return s;
  if (state == nullptr) return LCS_ERR_INVALID_ARG;
  if ((s = check_rows(&state->window)) != LCS_OK) return s;
  if ((s = check_rows(&state->new_rows)) != LCS_OK) return s;
  if (!same_layout(state->window, state->new_rows)) return LCS_ERR_SHAPE;
  if (state->window.num_rows < (int64_t)batch->num_seqs * LCSA_WINDOW) return LCS_ERR_SHAPE;
  return from_cuda(launch_window_commit(batch->cu_new, batch->seq_len, batch->num_seqs, batch->max_new,
                                        make_rows(state->new_rows), make_rows(state->window), dev_status,
                                        static_cast<cudaStream_t>(stream)));
}



lcs_status csa_index_topk(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale, const float* head_w,
                          int32_t heads, const lcs_index_keys* keys, const lcs_paging* paging, int32_t m, int32_t k,
                          int32_t flags, int32_t* out_idx, int32_t* out_cnt, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream) {
  IndexParams p;
  lcs_status s = index_common(batch, q_fp4, q_scale, heads, keys, paging, m, p);
  if (s != LCS_OK) return s;
  if (k < 1 || k > 4096) return LCS_ERR_UNSUPPORTED;
  if ((flags & ~(LCS_INDEX_RELU | LCS_INDEX_SCORE_ONLY | LCS_INDEX_SELECT_ONLY | LCS_INDEX_SPARE_SMS(0xFF))) != 0)
    return LCS_ERR_INVALID_ARG;
  const int sms = std::max(std::min(16, num_sms()), num_sms() - ((flags >> 8) & 0xFF));
  const bool score_only = (flags & LCS_INDEX_SCORE_ONLY) != 0, select_only = (flags & LCS_INDEX_SELECT_ONLY) != 0;
  if (score_only && select_only) return LCS_ERR_INVALID_ARG;
  if (!score_only && (out_idx == nullptr || out_cnt == nullptr)) return LCS_ERR_INVALID_ARG;
  const TopkWs w = topk_ws_layout(batch, p, keys->rank, m, k, sms);
  if (workspace == nullptr || workspace_bytes < w.total) return LCS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LCS_ERR_ALIGNMENT;
  p.head_w = head_w;
  p.relu = (flags & LCS_INDEX_RELU) ? 1 : 0;
  p.ld = index_ld(batch, m);
  p.status = dev_status;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int max_entries = batch->max_seq_len / m;
  cudaError_t e = cudaSuccess;
  if (w.fused) {
    p.top_k = k;
    p.cand_cap = w.plan.cap;
    p.runs.runs = w.plan.runs;
    p.runs.ticket = reinterpret_cast<int*>(ws + w.ticket);
    p.runs.cnt = reinterpret_cast<int*>(ws + w.cnt);
    p.runs.tau = reinterpret_cast<uint64_t*>(ws + w.tau);
    // (a scoring call on its own shares no threshold: the counters stay zero without a merge)
    p.runs.gthr = score_only || select_only ? nullptr : reinterpret_cast<uint64_t*>(ws + w.gthr);
    p.runs.keys = reinterpret_cast<uint64_t*>(ws + w.keys);
    p.runs.list_cap = w.plan.list_cap;
    p.out_idx = out_idx;
    p.out_cnt = out_cnt;
    if (select_only) return from_cuda(launch_topk_merge(p, w.plan, batch->max_new, st));
    p.merge_inline = (!score_only && w.plan.merge_inline) ? 1 : 0;
    e = launch_index_tc(p, w.plan, st);
    if (e != cudaSuccess || score_only || p.merge_inline) return from_cuda(e);
    return from_cuda(launch_topk_merge(p, w.plan, batch->max_new, st));
  }
  p.keys_out = reinterpret_cast<uint32_t*>(ws + w.keys);
  p.hist = reinterpret_cast<uint32_t*>(ws + w.hist);
  if (!select_only) {
    // the per-query histograms accumulate with atomics: clear them first
    e = cudaMemsetAsync(ws + w.hist, 0, (size_t)batch->total_new * kTopkHistBins * 4, st);
    if (e != cudaSuccess) return LCS_ERR_CUDA;
    e = launch_score_keys(p, keys->rank, batch->max_new, max_entries, st);
    if (e != cudaSuccess || score_only) return from_cuda(e);
  }
  e = launch_topk_select(p.keys_out, p.hist, p.ld, batch->cu_new, batch->seq_len, batch->num_seqs, batch->max_new,
                         m, k, out_idx, out_cnt, st);
  return from_cuda(e);
}

lcs_status csa_index_scores(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale, const float* head_w,
                            int32_t heads, const lcs_index_keys* keys, const lcs_paging* paging, int32_t m,
                            int32_t flags, float* out_scores, int64_t ld, int32_t* dev_status, void* stream) {
  IndexParams p;
  lcs_status s = index_common(batch, q_fp4, q_scale, heads, keys, paging, m, p);
  if (s != LCS_OK) return s;
  if ((flags & ~LCS_INDEX_RELU) != 0 || out_scores == nullptr) return LCS_ERR_INVALID_ARG;
  if (ld < batch->max_seq_len / m) return LCS_ERR_SHAPE;
  p.head_w = head_w;
  p.relu = (flags & LCS_INDEX_RELU) ? 1 : 0;
  p.ld = ld;
  p.scores_out = out_scores;
  p.status = dev_status;
  return from_cuda(launch_scores(p, batch, keys->rank, m, static_cast<cudaStream_t>(stream)));
}

size_t lcs_attend_workspace(const lcs_batch* batch, int32_t heads, int32_t dim, int32_t max_rows) {
  if (batch == nullptr) return 0;
  // the same size serves a CSA call (window apart), an HCA call (one list) and calls with values
  // (warp-MMA plan)
  return std::max({attend_ws_bytes(batch, heads, dim, plan_splits(batch, heads, dim, max_rows, true)),
                   attend_ws_bytes(batch, heads, dim, plan_splits(batch, heads, dim, max_rows, false)),
                   attend_ws_bytes(batch, heads, dim, plan_splits(batch, heads, dim, max_rows, false, false))});
}

lcs_status csa_attend(const lcs_batch* batch, const void* q, int32_t heads, const int32_t* topk_idx,
                      const int32_t* topk_cnt, int32_t k, int32_t m, const lcs_rows* entries, const lcs_paging* paging,
                      const lcs_state* state, const lcs_values* values, const float* sink, float softmax_scale,
                      void* out, float* out_lse, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      void* stream) {
  return csa_attend_part(batch, q, heads, topk_idx, topk_cnt, k, m, entries, paging, state, values, sink,
                         softmax_scale, out, out_lse, workspace, workspace_bytes, dev_status, stream, 0);
}

lcs_status csa_attend_window(const lcs_batch* batch, const void* q, int32_t heads, int32_t k, int32_t m,
                             const lcs_rows* entries, const lcs_paging* paging, const lcs_state* state,
                             const lcs_values* values, float softmax_scale, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream) {
  return csa_attend_part(batch, q, heads, nullptr, nullptr, k, m, entries, paging, state, values, nullptr,
                         softmax_scale, nullptr, nullptr, workspace, workspace_bytes, dev_status, stream, 1);
}

lcs_status csa_attend_topk(const lcs_batch* batch, const void* q, int32_t heads, const int32_t* topk_idx,
                           const int32_t* topk_cnt, int32_t k, int32_t m, const lcs_rows* entries,
                           const lcs_paging* paging, const lcs_state* state, const lcs_values* values,
                           const float* sink, float softmax_scale, void* out, float* out_lse, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return csa_attend_part(batch, q, heads, topk_idx, topk_cnt, k, m, entries, paging, state, values, sink,
                         softmax_scale, out, out_lse, workspace, workspace_bytes, dev_status, stream, 2);
}

lcs_status hca_attend(const lcs_batch* batch, const void* q, int32_t heads, int32_t m, const lcs_rows* entries,
                      const lcs_paging* paging, const lcs_state* state, const lcs_values* values, const float* sink,
                      float softmax_scale, void* out, float* out_lse, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream) {
  if (m <= 0 || m > 128) return LCS_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(sink) & 3u) return LCS_ERR_ALIGNMENT;
  AttendParams p;
  lcs_status s = attend_common(batch, q, heads, entries, paging, state, values, out, workspace, workspace_bytes,
                               batch ? batch->max_seq_len / m + LCSA_WINDOW : 0, p, false);
  if (s != LCS_OK) return s;
  p.m = m;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.sink = sink;
  p.out_lse = out_lse;
  p.status = dev_status;
  return from_cuda(launch_attend(p, entries->dim, entries->format, batch->total_new, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
