// Lightning-indexer scores and top-k on the tcgen05 tensor cores for batches with a few queries
// per sequence (decode, short speculative runs).
//
// Defined by: m.x-techcon.com/article/133366, section 2, CSA step 2 (a low-rank indexer scores
// every compressed entry, each query keeps its top-k) and section 4 "FP4量化感知训练" (the
// indexer's QK path runs in FP4).  Same arithmetic as the warp-MMA scorer in indexer.cu:
//   score(q, j) = sum_h w[q,h] * phi( sum_blk 2^(eq[q,h,blk] + ek[j,blk]) * dot_blk(q_h, k_j) ).
//
// Layout of the work.  A persistent, warp-specialised CTA scans a contiguous run of 128-entry
// tiles of one sequence for all of that sequence's queries (QPS <= 4), through a ring of
// shared-memory stages:
//   warps 8-9 (producers, alternating tiles) stream tiles: one lane per page issues a TMA copy
//                      of the page's codes as they are stored, two E2M1 codes a byte, with the
//                      64-byte swizzle -- each entry's 128 codes occupy one 64-byte shared-memory
//                      row, the K-major operand form of the block-scaled kind::mxf4 MMA -- and
//                      every lane copies 16 bytes of block scales with cp.async;
//   warp 10 (MMA)      issues two K = 64 MMAs per tile into one of the tensor-memory accumulators
//                      and commits them to that accumulator's barrier;
//   warps 0-7          (one thread per entry = per TMEM lane, two warps per lane quadrant taking
//                      the two tiles of a tile pair) read the accumulator, release it and form
//                      the scores.
// The grid is one wave: about (SMs x resident CTAs) / sequences CTAs per sequence.
//
// The MMA: A = 128 entries x 128 codes, B = N rows built from the queries, where row
// (blk, q, h) holds query q's head-h codes inside block blk and zeros elsewhere.  Two
// kind::mxf4 MMAs of K = 64 accumulate into D = 128 x N fp32 in tensor memory with every scale
// factor 2^0 (UE8M0 127, eight tensor-memory columns written once); because every B row is zero
// outside its block, column (blk, q, h) of D is exactly that block's partial dot product (a sum of
// 32 products of E2M1 values: multiples of 1/4 below 2^11, exact in fp32).  Block scales and head
// weights are applied afterwards in fp32, as in the warp-MMA scorer, so that every score is the
// same fp32 arithmetic whatever the scales (the packed operand halves the shared memory a tile
// needs, which doubles the tiles in flight).
//
// Top-k, fused into the epilogue (FUSED = true).  Each query's candidates are 64-bit keys
// (score key << 32 | ~j) in a shared-memory buffer of cap >= k + k/8 + 256 keys: a score enters
// when its key beats the query's threshold (no key below it can be among the k largest of the
// run, nor of the sequence).  After every tile pair the epilogue warps meet at a named barrier; a
// buffer past cap - 256 is cut by a radix selection that stops at a digit bin leaving k to
// k + k/8 keys, whose lower edge becomes the threshold -- published to the query's other runs,
// whose thresholds are just as valid (each is at most the query's k-th largest key).  At the end
// of its run a CTA writes its keys at or above a threshold that k to k + k/4 of them reach (the
// same radix selection, stopped at a digit bin), ascending in j, their count and that threshold
// to the workspace; the sequence's last CTA to finish (a ticket counter, left at zero again)
// merges the runs' lists: the largest of the runs' thresholds bounds the selection from below, the
// k-th largest key comes from the exact radix selection, and the staged lists are read out in
// ascending j.  A separate merge kernel does the same when the scoring phase runs
// alone or the lists do not fit the CTA's shared memory.  FUSED = false writes the fp32 scores
// themselves (csa_index_scores).
#include <algorithm>

#include "kernels.cuh"
#include "select.cuh"
#include "sm100.cuh"

namespace lcsa {

namespace {

constexpr int kTile = 128;          // entries per MMA tile (M)
// shared-memory ring depth (tiles in flight per CTA): the shallow ring leaves room for candidate
// buffers that take a whole run without a compaction; the deep one, for long runs with long lists,
// lets the last CTA stage every run's list in the idle ring
constexpr int kStagesShallow = 6;
constexpr int kStagesDeep = 10;
constexpr int kAcc = 8;             // tensor-memory accumulators at most (the MMA runs up to 8 tiles ahead)
constexpr int kSfCols = 8;          // tensor-memory columns of the (unit) scale factors
constexpr int kMaxPages = 8192;     // block-table entries a CTA's run may span
constexpr int kRowBytes = 64;       // shared-memory bytes of one entry's 128 codes (packed)
constexpr int kPackedRowBytes = 64; // global bytes of the same codes
constexpr int kATileBytes = kTile * kRowBytes;
constexpr int kEpiWarps = 8;        // two per TMEM lane quadrant, the two tiles of a pair
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kProdWarps = 2;       // producer warps, alternating tiles
constexpr int kThreads = kEpiThreads + 32 * kProdWarps + 32;
constexpr int kCandPerThread = 8;  // keys a thread holds in registers in one block of a compaction
constexpr int kEpiBarrier = 1;      // named barrier of the epilogue warps
constexpr int kMaxRuns = 256;       // CTAs per sequence (run lists a merge reads)

// block-scale ring: tile i's scales are copied once stage i % kStages is free (the MMA of tile
// i - kStages is done, so the epilogue has read tile i - kStages - accumulators); they are read
// by the epilogue of tile i, so kStages + kAcc tiles' scales can be live at once
template <int QH, int QPS, int ST>
struct TcSmem {
  static constexpr int kStages = ST;
  static constexpr int kScaleSlots = ST + kAcc;
  static constexpr int N = 4 * QH;                            // MMA N: (block, query-head) columns
  // the fixed part first
  static constexpr int kB = 0;                                // N x 64 B (1024-aligned)
  static constexpr int kScale = kB + N * kRowBytes;           // kScaleSlots x 128 x 4 B
  static constexpr int kQs = kScale + kScaleSlots * kTile * 4;  // f32 [QH][4] q block scales
  static constexpr int kHw = kQs + QH * 4 * 4;                // f32 [QH] head weights
  static constexpr int kQw = kHw + QH * 4;                    // f32 [QH][4] q block scale x head weight
  static constexpr int kBar = (kQw + QH * 4 * 4 + 7) / 8 * 8;  // u64 full/empty[kStages], accf/acce[kAcc], drain
  static constexpr int kArmed = kBar + (2 * kStages + 2 * kAcc + 1) * 8;   // int [kStages] last tile armed
  static constexpr int kMisc = kArmed + kStages * 4 + 4;      // tmem base, abort flag, last-CTA flag
  // (16-byte aligned from here on: the selection scratch holds 8-byte fields)
  static constexpr int kThr = (kMisc + 16 + 15) / 16 * 16;    // u64 [QPS] thresholds
  static constexpr int kCnt = kThr + QPS * 8;                 // int [QPS] candidate counts
  static constexpr int kSelEpi = (kCnt + QPS * 4 + 15) / 16 * 16;   // SelScratch<kEpiThreads>
  static_assert(alignof(SelScratch<kThreads>) <= 16 && alignof(SelScratch<kEpiThreads>) <= 16, "scratch alignment");
  static constexpr int kCand = (kSelEpi + (int)sizeof(SelScratch<kEpiThreads>) + 15) / 16 * 16;   // u64 [QPS][cap]
  // then the ring of kStages x 8 KB (1024-aligned) right after the candidate buffers, then the
  // run's page table: int [pages].  After the scan the ring is idle: its tail holds the whole CTA's
  // selection scratch, the merge's run offsets and a 2048-bin histogram, its head the run bitmap
  // (final selection); the merge stages the run lists from the (idle) candidate buffers on through
  // the ring up to the histogram.
  static constexpr int kRingBytes = kStages * kATileBytes;
  static constexpr int kRunOffR = (kRingBytes - 4 * (kMaxRuns + 4)) / 16 * 16;              // int [runs + 1]
  static constexpr int kSelAllR = (kRunOffR - (int)sizeof(SelScratch<kThreads>)) / 16 * 16;  // SelScratch<kThreads>
  static constexpr int kHistR = kSelAllR - 2048 * 4;                                       // u32 [2048]
  __host__ __device__ static constexpr int ring_off(bool fused, int cap) {
    return (kCand + (fused ? QPS * cap * 8 : 0) + 1023) / 1024 * 1024;
  }
  static size_t bytes(bool fused, int cap, int pages) {
    return (size_t)ring_off(fused, cap) + kRingBytes + (size_t)pages * 4 + 1024;
  }
  static size_t stage_bytes(int cap) { return (size_t)(ring_off(true, cap) + kHistR - kCand); }
};

// accumulators of N columns: 8 while they and the scale factors fit 256 columns, else 7 (which
// keeps 32 query-head columns at two CTAs an SM and 64 within the 512 columns)
__host__ __device__ constexpr int acc_for(int n) { return 8 * n + kSfCols <= 256 ? 8 : 7; }

__host__ __device__ constexpr uint32_t tmem_cols_for(int n) {
  const int c = acc_for(n) * n + kSfCols;
  return c <= 32 ? 32 : (c <= 64 ? 64 : (c <= 128 ? 128 : (c <= 256 ? 256 : 512)));
}

}  // namespace

// The run's selected keys (those >= tau of buf[0..n)), written to dst in ascending entry index:
// a bitmap over the run's entries [j0, j0 + 32*words) gives every key its rank by position
// (keys of the run lie in that range).  Group of NT threads; bitmap: `words` words and prefix:
// `words` ints of shared memory.  Returns the number written.
template <int NT, int ID>
__device__ int write_run_sorted(const uint64_t* buf, int n, uint64_t tau, int j0, int words, uint32_t* bitmap,
                                int* prefix, uint64_t* dst, SelScratch<NT>& sc) {
  const int tid = threadIdx.x;
  for (int w = tid; w < words; w += NT) bitmap[w] = 0u;
  group_sync<NT, ID>();
  for (int x = tid; x < n; x += NT) {
    const uint64_t u = buf[x];
    if (u >= tau) {
      const uint32_t rj = ~(uint32_t)u - (uint32_t)j0;
      atomicOr(&bitmap[rj >> 5], 1u << (rj & 31u));
    }
  }
  group_sync<NT, ID>();
  // exclusive prefix of the words' bit counts: thread t sums words [t*wpt, (t+1)*wpt)
  const int wpt = (words + NT - 1) / NT;
  const int w0 = min(words, tid * wpt), w1 = min(words, w0 + wpt);
  int mine = 0;
  for (int w = w0; w < w1; ++w) mine += __popc(bitmap[w]);
  int tot;
  int run = group_scan_incl<NT, ID>(mine, sc.warp_tot, &tot) - mine;
  for (int w = w0; w < w1; ++w) {
    prefix[w] = run;
    run += __popc(bitmap[w]);
  }
  group_sync<NT, ID>();
  for (int x = tid; x < n; x += NT) {
    const uint64_t u = buf[x];
    if (u >= tau) {
      const uint32_t rj = ~(uint32_t)u - (uint32_t)j0;
      const int w = (int)(rj >> 5);
      dst[prefix[w] + __popc(bitmap[w] & ((1u << (rj & 31u)) - 1u))] = u;
    }
  }
  group_sync<NT, ID>();
  return tot;
}

// The merge of one query's run lists into its top-k (the scorer's last CTA of a query group, or
// the merge kernel).  Group of NT threads (ID 0: the whole CTA).  Every run list is sorted by entry
// index and the runs cover increasing index ranges, so the lists read one after the other are
// sorted too: they are staged in shared memory (stage: room for stage_cap keys), the k-th largest
// key is selected, and the staged keys at or above it are read out in that order.  Every run
// recorded a threshold at most the query's k-th largest key (at least k of the run's keys, or all
// of them, are at or above it), with all of its keys at or above it in its list; the largest of
// those bounds the selection from below (the selection reads the stage and leaves out the keys
// under the bound: with a few runs a query nearly all staged keys pass it, so gathering the
// candidates first would cost a pass and save none).  N: visible entries of the query; run_off:
// runs + 1 ints of shared memory; hist: 1 << BITS counters of shared memory.
template <int NT, int ID, int BITS>
__device__ void merge_query_topk(const TopkRuns& tr, long long q, int N, int k, uint64_t* stage, int stage_cap,
                                 int* run_off, uint32_t* hist, int32_t* out_idx,
                                 int32_t* out_cnt, SelScratch<NT>& sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* out = out_idx + q * k;
  if (N <= k) {   // every visible entry
    for (int j = tid; j < k; j += NT) out[j] = j < N ? j : -1;
    if (tid == 0) out_cnt[q] = N;
    return;
  }
  const int* cnts = tr.cnt + q * tr.runs;
  const int lcap = tr.list_cap;
  const unsigned long long* keys = reinterpret_cast<const unsigned long long*>(tr.keys) + q * (long long)tr.runs * lcap;
  // list offsets in the stage, and the bound: the largest threshold of the runs (runs <= 256 <= NT)
  uint64_t bound;
  {
    const int c = tid < tr.runs ? min(__ldcg(cnts + tid), lcap) : 0;
    unsigned long long t = tid < tr.runs ? __ldcg(reinterpret_cast<const unsigned long long*>(tr.tau) + q * tr.runs + tid)
                                         : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, t, o);
      t = y > t ? y : t;
    }
    if (lane == 0) sc.span[warp] = t;
    int tot;
    const int incl = group_scan_incl<NT, ID>(c, sc.warp_tot, &tot);   // (its barriers publish span)
    if (tid < tr.runs) run_off[tid] = incl - c;
    if (tid == 0) run_off[tr.runs] = tot;
    unsigned long long bmax = 0ull;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) bmax = sc.span[w] > bmax ? sc.span[w] : bmax;
    bound = bmax;
  }
  group_sync<NT, ID>();
  const int total = min(run_off[tr.runs], stage_cap);   // (the host sizes the stage for every list)
  // stage the lists, a warp per run, by 8-byte asynchronous copies (every copy in flight at once,
  // no registers held)
  for (int r = warp; r < tr.runs; r += NT / 32) {
    const int o = run_off[r];
    const int c = min(run_off[r + 1], total) - o;
    const unsigned long long* src = keys + (long long)r * lcap;
    for (int x = lane; x < c; x += 32)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(stage + o + x)), "l"(src + x) : "memory");
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  group_sync<NT, ID>();
  // (fewer than k keys only when the scoring gave up on a bounded wait: take them all)
  const uint64_t tau = total > k ? kth_largest_key<NT, ID, BITS>(stage, total, k, sc, hist, bound) : 0ull;
  // ascending read-out: thread t takes stage positions [t*ppt, (t+1)*ppt)
  const int ppt = (total + NT - 1) / NT;
  const int x0 = min(total, tid * ppt), x1 = min(total, x0 + ppt);
  int mine = 0;
  for (int x = x0; x < x1; ++x) mine += stage[x] >= tau ? 1 : 0;
  int tot;
  int pos = group_scan_incl<NT, ID>(mine, sc.warp_tot, &tot) - mine;
  for (int xb = x0; xb < x1; xb += 8) {   // (8 keys read before their stores: the loads overlap)
    uint64_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = xb + u < x1 ? stage[xb + u] : 0ull;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (xb + u < x1 && v[u] >= tau) {
        if (pos < k) out[pos] = (int32_t)~(uint32_t)v[u];
        ++pos;
      }
  }
  for (int j = tot + tid; j < k; j += NT) out[j] = -1;   // (tot == k for exact selections)
  if (tid == 0) out_cnt[q] = min(tot, k);
  group_sync<NT, ID>();
}

// grid: (runs, query groups, num_seqs); block kThreads.  CTA (x, g, b) scans tiles
// [x*tiles_per_cta, (x+1)*tiles_per_cta) of sequence b (clipped to its visible entries) for the
// sequence's queries g*QPS .. g*QPS + QPS - 1.
template <int HI, int QH, bool FUSED, int ST>
__global__ void __launch_bounds__(kThreads, QH >= 16 ? 1 : 2) index_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                           const __grid_constant__ CUtensorMap tmap_t, IndexParams p,
                                                           int tiles_per_cta) {
  constexpr int QPS = QH / HI;
  using L = TcSmem<QH, QPS, ST>;
  constexpr int kStages = L::kStages;
  constexpr int kScaleSlots = L::kScaleSlots;
  constexpr int N = L::N;
  constexpr uint32_t kCols = tmem_cols_for(N);
  constexpr int kAccN = acc_for(N);
  constexpr uint32_t kIdesc = idesc_mxf4(kTile, N);  // E2M1 x E2M1 (unit block scales) -> f32, M = 128
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int qg0 = blockIdx.y * QPS;                // the group's first query within the sequence
  const int qn = min(sp.qn - qg0, QPS);
  if (qn <= 0) return;   // (every CTA of the query group returns here: no ticket is taken)
  const long long qrow0 = (long long)sp.q0 + qg0;  // its row in the batch
  const int n0 = sp.n0() + qg0;                    // its position
  const int mshift = 31 - __clz(p.m);
  const int nmax = (n0 + qn) >> mshift;          // visible entries of the sequence's last query
  const int t_begin = blockIdx.x * tiles_per_cta;
  const int t_end = min((nmax + kTile - 1) / kTile, t_begin + tiles_per_cta);
  const int nt = max(0, t_end - t_begin);
  const int k = p.top_k;
  const int cap = p.cand_cap;
  const int ring_off = L::ring_off(FUSED, cap);   // the ring after the candidate buffers
  SelScratch<kThreads>& sel_all = *reinterpret_cast<SelScratch<kThreads>*>(smem + ring_off + L::kSelAllR);
  uint64_t* thr_s = reinterpret_cast<uint64_t*>(smem + L::kThr);
  int* cnt_s = reinterpret_cast<int*>(smem + L::kCnt);
  uint64_t* cand_s = reinterpret_cast<uint64_t*>(smem + L::kCand);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 8);
  if (nt == 0) {
    if constexpr (FUSED) {
      // no tiles in this run (ragged batch): an empty candidate list, and the ticket still counts it
      for (int qi = tid; qi < qn; qi += kThreads) {
        p.runs.cnt[(qrow0 + qi) * p.runs.runs + blockIdx.x] = 0;
        p.runs.tau[(qrow0 + qi) * p.runs.runs + blockIdx.x] = 0ull;
      }
    } else {
      return;
    }
  }
  const int epb = p.paging.epb;
  const int eshift = 31 - __clz(epb);
  const int page0 = (t_begin * kTile) >> eshift;
  const int npages = nt > 0 ? ((min(nmax, t_end * kTile) - 1) >> eshift) - page0 + 1 : 0;  // <= kMaxPages (host)

  float* qs_s = reinterpret_cast<float*>(smem + L::kQs);
  float* hw_s = reinterpret_cast<float*>(smem + L::kHw);
  float* qw_s = reinterpret_cast<float*>(smem + L::kQw);
  int* pages_s = reinterpret_cast<int*>(smem + ring_off + L::kRingBytes);
  int* armed_s = reinterpret_cast<int*>(smem + L::kArmed);
  const uint32_t bar_full = sbase + L::kBar;
  const uint32_t bar_empty = bar_full + kStages * 8;
  const uint32_t bar_accf = bar_empty + kStages * 8;
  const uint32_t bar_acce = bar_accf + kAcc * 8;
  const uint32_t bar_drain = bar_acce + kAcc * 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  const uint32_t polls = p.wait_polls;

  if (nt > 0) {
    if (tid == kEpiThreads) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(bar_full + 8 * i, 1);    // the expect-tx arrival (codes and scales: transaction bytes)
        mbar_init(bar_empty + 8 * i, 1);   // the MMA commit
        armed_s[i] = -1;
      }
      for (int i = 0; i < kAcc; ++i) {
        mbar_init(bar_accf + 8 * i, 1);
        mbar_init(bar_acce + 8 * i, 4);
      }
      mbar_init(bar_drain, 1);
      *abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_t);
    }
    if (FUSED && tid < QPS) {
      thr_s[tid] = 0ull;
      cnt_s[tid] = 0;
    }
    // the physical block of every page the run touches, copied by every thread at once (the
    // producer lane that reads an entry checks it)
    for (int i = tid; i < npages; i += kThreads) {
      const int blk = page0 + i;
      if (blk < p.paging.max_blocks)
        cp_async4(pages_s + i, p.paging.table + (long long)b * p.paging.max_blocks + blk);
      else
        pages_s[i] = -1;
    }
    cp_async_commit();
    __syncthreads();

    if (warp == kEpiWarps) {
      tmem_alloc(sbase + L::kMisc, kCols);
    } else if (warp < kEpiWarps) {
      // ---- B operand: row n = blk*QH + c, c = qi*HI + h; the 16-byte chunk blk of its 64 bytes
      //      holds block blk's 32 packed codes (64-byte swizzle: chunk ch of row n at ch ^ (n/2 % 4))
      for (int idx = tid; idx < N * 4; idx += kEpiThreads) {
        const int n = idx >> 2, ch = idx & 3;
        const int blk = n / QH, c = n % QH;
        const int qi = c / HI, h = c % HI;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ch == blk && qi < qn) {
          const long long qrow = (qrow0 + qi) * HI + h;
          const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q_fp4 + qrow * 64 + ch * 16);
          v = make_uint4(src[0], src[1], src[2], src[3]);
        }
        const int phys_ch = ch ^ ((n >> 1) & 3);
        *reinterpret_cast<uint4*>(smem + L::kB + n * kRowBytes + phys_ch * 16) = v;
      }
      for (int idx = tid; idx < QH * 4; idx += kEpiThreads) {
        const int c = idx >> 2, blk = idx & 3;
        const int qi = c / HI, h = c % HI;
        const float qs = qi < qn ? ue8m0_to_f32(p.q_scale[((qrow0 + qi) * HI + h) * 4 + blk]) : 0.0f;
        qs_s[idx] = qs;
        // powers of two times the head weight: exact
        qw_s[idx] = qi < qn ? qs * (p.head_w ? p.head_w[(qrow0 + qi) * HI + h] : 1.0f) : 0.0f;
      }
      for (int c = tid; c < QH; c += kEpiThreads) {
        const int qi = c / HI, h = c % HI;
        hw_s[c] = qi < qn ? (p.head_w ? p.head_w[(qrow0 + qi) * HI + h] : 1.0f) : 0.0f;
      }
      fence_proxy_async_smem();
    }
    cp_async_wait<0>();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // do the run's pages follow one another in the cache (every one mapped and inside the key rows)?
    bool contig_mine = true;
    for (int i = tid; i < npages; i += kThreads) {
      const int ph = pages_s[i];
      contig_mine = contig_mine && ph >= 0 && ph == pages_s[0] + i && (long long)(ph + 1) * epb <= p.k_rows;
    }
    // the scale factors of every MMA, 2^0: written once by warps 0-3 (their tensor-memory lanes)
    if (warp < 4) {
      const uint32_t tm_sf = tmem + kAccN * N + ((uint32_t)(warp * 32) << 16);
      tmem_st4_fill(tm_sf, 0x7F7F7F7Fu);
      tmem_st4_fill(tm_sf + 4, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
    tc_fence_before_sync();
    const bool run_contig = __syncthreads_and(contig_mine ? 1 : 0) != 0;
    tc_fence_after_sync();

    if (warp >= kEpiWarps && warp < kEpiWarps + kProdWarps) {
      // ---- producer warps (tile i by producer warp i % kProdWarps): stage i % kStages receives
      //      tile t_begin + i: the codes by tensor copies (the TMA lays them out in the MMA operand
      //      form) and the block scales by bulk copies, all counted in the stage barrier's
      //      transaction bytes.  A run whose pages are consecutive blocks of the cache (checked
      //      once) takes one thread a tile: one copy of 128 rows and one of their scales; otherwise
      //      lane p copies page p.
      for (int i = warp - kEpiWarps; i < nt; i += kProdWarps) {
        const int s = i % kStages;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(bar_empty + 8 * s, ((i / kStages) & 1) ^ 1, p.status, abort_flag, polls);
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
        const int e0 = (t_begin + i) * kTile;
        const int rows = min(kTile, ((min(nmax, e0 + kTile) - e0 + epb - 1) >> eshift) << eshift);  // whole pages
        const uint32_t bar = bar_full + 8 * s;
        const uint32_t a_dst = sbase + ring_off + s * kATileBytes;
        const uint32_t s_dst = sbase + L::kScale + (i % kScaleSlots) * kTile * 4;
        const int npg = rows >> eshift;
        if (run_contig) {
          if (lane == 0) {
            const int p0 = pages_s[(e0 >> eshift) - page0];
            armed_s[s] = i;
            mbar_arrive_expect_tx(bar, rows * (kPackedRowBytes + 4));
            if (rows == kTile) {
              tma_load_2d(a_dst, &tmap_t, 0, p0 * epb, bar);
            } else {
              for (int pg = 0; pg < npg; ++pg) tma_load_2d(a_dst + (pg << eshift) * kRowBytes, &tmap_k, 0, (p0 + pg) * epb, bar);
            }
            bulk_load(s_dst, p.k_scale + (long long)p0 * epb * 4, rows * 4, bar);
          }
        } else {
          int phys = lane < npg ? pages_s[((e0 >> eshift) - page0) + lane] : -1;
          if (lane < npg && (phys < 0 || (long long)(phys + 1) * epb > p.k_rows)) {
            report(p.status, LCS_ERR_DEVICE_GUARD);   // unmapped, or outside the key rows
            phys = -1;
          }
          const uint32_t valid = __ballot_sync(0xffffffffu, phys >= 0);
          if (lane == 0) {
            armed_s[s] = i;
            mbar_arrive_expect_tx(bar, __popc(valid) * epb * (kPackedRowBytes + 4));
          }
          __syncwarp();
          if (phys >= 0) {
            tma_load_2d(a_dst + (lane << eshift) * kRowBytes, &tmap_k, 0, phys * epb, bar);
            bulk_load(s_dst + (lane << eshift) * 4, p.k_scale + (long long)phys * epb * 4, epb * 4, bar);
          }
        }
      }
    } else if (warp == kEpiWarps + kProdWarps) {
      if (lane == 0) {
        // ---- MMA issuer: tile i -> accumulator i % kAccN
        const uint64_t bdesc = smem_desc_sw64(sbase + L::kB);
        const uint32_t tm_sf = tmem + kAccN * N;
        bool issued = false;
        for (int i = 0; i < nt; ++i) {
          const int s = i % kStages, a = i % kAccN;
          if (!mbar_wait(bar_full + 8 * s, (i / kStages) & 1, p.status, abort_flag, polls)) break;
          if (!mbar_wait(bar_acce + 8 * a, ((i / kAccN) & 1) ^ 1, p.status, abort_flag, polls)) break;
          tc_fence_after_sync();
          const uint64_t adesc = smem_desc_sw64(sbase + ring_off + s * kATileBytes);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb)   // K = 64 codes per MMA: 32 shared-memory bytes per step
            tc_mma_mxf4(tmem + a * N, adesc + 2 * kb, bdesc + 2 * kb, kIdesc, tm_sf, tm_sf + 4, kb > 0 ? 1u : 0u);
          tc_commit(bar_accf + 8 * a);
          tc_commit(bar_empty + 8 * s);   // the stage is free once these MMAs have read it
          issued = true;
        }
        // every MMA issued here has completed before the CTA releases tensor memory
        if (issued && *abort_flag) {
          tc_commit(bar_drain);
          mbar_wait(bar_drain, 0, nullptr, nullptr, kWaitPolls);
        }
      }
      __syncwarp();
    } else {
      // ---- epilogue: tile pair ip = tiles 2ip (warps 0-3) and 2ip+1 (warps 4-7); warp w reads
      //      TMEM lanes 32*(w%4).. (its entries)
      const int quad = warp & 3, par = warp >> 2;
      // (the query's block scales and head weights are read from shared memory where they are
      // used: broadcast reads, registers kept for the accumulator columns)
      int nq[QPS];
#pragma unroll
      for (int qi = 0; qi < QPS; ++qi) nq[qi] = qi < qn ? (n0 + qi + 1) >> mshift : 0;
      const int row = quad * 32 + lane;
      SelScratch<kEpiThreads>& sel = *reinterpret_cast<SelScratch<kEpiThreads>*>(smem + L::kSelEpi);
      bool alive = true;
      const bool share = FUSED && p.runs.gthr != nullptr;
      // a warp takes kPerWarp tiles an iteration (the two warp groups alternate) and the warps meet
      // once an iteration (measured: two tiles a warp was no faster and needs more candidate room)
      constexpr int kPerWarp = 1;
      constexpr int kIter = 2 * kPerWarp;
      // the scores of tile i (accumulator columns d, the entries' block-scale word sc)
      auto score_tile = [&](const uint32_t (&d)[N], uint32_t sc, int i) {
        // 2^(e-127) for the four UE8M0 bytes (e = 0 gives the subnormal 2^-127)
        float ksc[4];
        ksc[0] = __uint_as_float(max((sc << 23) & 0x7F800000u, 0x00400000u));
        ksc[1] = __uint_as_float(max((sc << 15) & 0x7F800000u, 0x00400000u));
        ksc[2] = __uint_as_float(max((sc << 7) & 0x7F800000u, 0x00400000u));
        ksc[3] = __uint_as_float(max((sc >> 1) & 0x7F800000u, 0x00400000u));
        const int j = (t_begin + i) * kTile + row;
#pragma unroll
        for (int qi = 0; qi < QPS; ++qi) {
          float score;
          if (!p.relu) {
            // phi = identity: sum over heads inside each block first (every term exact)
            float tb[4];
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
              float t = 0.0f;
#pragma unroll
              for (int h = 0; h < HI; ++h)
                t = fmaf(__uint_as_float(d[blk * QH + qi * HI + h]), qw_s[(qi * HI + h) * 4 + blk], t);
              tb[blk] = t;
            }
            score = fmaf(tb[3], ksc[3], fmaf(tb[2], ksc[2], fmaf(tb[1], ksc[1], tb[0] * ksc[0])));
          } else {
            float sh[HI];
#pragma unroll
            for (int h = 0; h < HI; ++h) {
              const int c = qi * HI + h;
              float acc = 0.0f;
#pragma unroll
              for (int blk = 0; blk < 4; ++blk)
                acc = fmaf(__uint_as_float(d[blk * QH + c]), ksc[blk] * qs_s[c * 4 + blk], acc);
              sh[h] = fmaxf(acc, 0.0f) * hw_s[c];
            }
#pragma unroll
            for (int w = 1; w < HI; w <<= 1)
#pragma unroll
              for (int h = 0; h < HI; h += 2 * w) sh[h] = sh[h] + sh[h + w];
            score = sh[0];
          }
          const bool vis = j < nq[qi];
          if constexpr (FUSED) {
            const uint64_t key = ((uint64_t)score_key(score) << 32) | (uint64_t)(~(uint32_t)j);
            warp_append(vis && key > thr_s[qi], key, cand_s + qi * cap, cnt_s + qi);
          } else {
            if (vis) p.scores_out[(qrow0 + qi) * p.ld + j] = score;
          }
        }
      };
      // the threshold the query's other runs have reached: read in one iteration and taken at the
      // end of the next, so that no iteration waits for the load (an older value is as valid)
      uint64_t gload = 0ull;
      for (int i0 = 0; i0 < nt; i0 += kIter) {
        const uint64_t gnext = gload;
        if (share && tid < qn) gload = __ldcg(reinterpret_cast<const unsigned long long*>(p.runs.gthr) + qrow0 + tid);
        uint32_t d[kPerWarp][N];
        bool have[kPerWarp];
#pragma unroll
        for (int u = 0; u < kPerWarp; ++u) {
          const int i = i0 + par + 2 * u;
          have[u] = i < nt && alive;
          if (have[u]) {
            const int a = i % kAccN;
            bool ok = mbar_wait(bar_accf + 8 * a, (i / kAccN) & 1, p.status, abort_flag, polls);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
              alive = false;
              have[u] = false;
            } else {
              tc_fence_after_sync();
#pragma unroll
              for (int c16 = 0; c16 < N / 16; ++c16)
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + a * N + c16 * 16,
                          *reinterpret_cast<uint32_t(*)[16]>(&d[u][c16 * 16]));
            }
          }
        }
        tmem_ld_wait();
        uint32_t sc[kPerWarp];
#pragma unroll
        for (int u = 0; u < kPerWarp; ++u)
          sc[u] = have[u] ? *reinterpret_cast<const uint32_t*>(
                                smem + L::kScale + (((i0 + par + 2 * u) % kScaleSlots) * kTile + row) * 4)
                          : 0u;
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0)
#pragma unroll
          for (int u = 0; u < kPerWarp; ++u)
            if (have[u]) mbar_arrive(bar_acce + 8 * ((i0 + par + 2 * u) % kAccN));
#pragma unroll
        for (int u = 0; u < kPerWarp; ++u)
          if (have[u]) score_tile(d[u], sc[u], i0 + par + 2 * u);
        if constexpr (FUSED) {
          // any run's threshold is at most the query's k-th largest key: a larger one from another
          // run filters this run's later keys too
          if (share && tid < qn && gnext > thr_s[tid]) thr_s[tid] = gnext;
          // the iteration's tiles are in: cut buffers that could not take another iteration
          group_sync<kEpiThreads, kEpiBarrier>();
#pragma unroll 1
          for (int qi = 0; qi < qn; ++qi) {
            const int n = cnt_s[qi];
            if (n <= cap - kIter * kTile) continue;    // uniform: read after the barrier
            uint64_t* buf = cand_s + qi * cap;
            // a threshold with k to k + k/8 of the buffer's keys at or above it (no more than the
            // buffer can keep while taking another pair), or the current one when fewer than k
            // keys pass that: every later key below it has k larger ones
            const uint64_t lo = thr_s[qi];
            const SelResult r = select_top<kEpiThreads, kEpiBarrier, 8>(buf, n, k, k >> 3, sel, sel.hist, lo);
            const uint64_t tau = r.tau > lo ? r.tau : lo;
            const int kept = compact_keys_ge<kEpiThreads, kEpiBarrier, kCandPerThread>(buf, n, tau, sel);
            if (tid == 0) {
              cnt_s[qi] = kept;
              thr_s[qi] = tau;
              // published to the query's other runs (theirs reach this run through the shared
              // threshold's read an iteration ahead: nothing waits for the atomic)
              if (share) atomicMax(reinterpret_cast<unsigned long long*>(p.runs.gthr) + qrow0 + qi, (unsigned long long)tau);
            }
            group_sync<kEpiThreads, kEpiBarrier>();
          }
        }
      }
    }
    tc_fence_before_sync();
    __syncthreads();
    // the scan is done: a programmatic dependent (the attention over the selected entries) may
    // start its own prologue on the SMs the scan leaves
    grid_launch_dependents();
    if (warp == kEpiWarps) {
      tc_fence_after_sync();
      tmem_dealloc(tmem, kCols);
    } else if (tid == kEpiThreads + 32 && *abort_flag) {
      // TMA copies still in flight after an abort land before the CTA leaves
      for (int s = 0; s < kStages; ++s)
        if (armed_s[s] >= 0) mbar_wait(bar_full + 8 * s, (armed_s[s] / kStages) & 1, nullptr, nullptr, kWaitPolls);
    }
    if constexpr (!FUSED) return;
    // ---- the run's k largest keys -> workspace, in ascending entry index (the ring is idle now:
    //      it holds the bitmap of the run's entries and its word prefixes)
    __syncthreads();
    const int words = nt * (kTile / 32);
    uint32_t* run_bits = reinterpret_cast<uint32_t*>(smem + ring_off);
    int* run_prefix = reinterpret_cast<int*>(smem + ring_off + words * 4);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + ring_off + L::kHistR);
#pragma unroll 1
    for (int qi = 0; qi < qn; ++qi) {
      const int n = cnt_s[qi];
      const uint64_t* buf = cand_s + qi * cap;
      // the run's list: its keys at or above a digit bin's lower edge with k to list_cap keys at or
      // above it, or all of them at or above the current threshold when fewer pass it (the buffer
      // holds every key of the run at or above that threshold); the merge selects exactly
      const uint64_t lo = thr_s[qi];
      uint64_t tau = lo;
      if (n > 0) {
        const SelResult r = select_top<kThreads, 0, 11>(buf, n, k, p.runs.list_cap - k, sel_all, hist, lo);
        tau = r.tau > lo ? r.tau : lo;
      }
      const long long q = qrow0 + qi;
      uint64_t* dst = p.runs.keys + (q * p.runs.runs + blockIdx.x) * (long long)p.runs.list_cap;
      const int w = write_run_sorted<kThreads, 0>(buf, n, tau, t_begin * kTile, words, run_bits, run_prefix, dst,
                                                   sel_all);
      if (tid == 0) {
        p.runs.cnt[q * p.runs.runs + blockIdx.x] = w;
        p.runs.tau[q * p.runs.runs + blockIdx.x] = tau;
      }
    }
  }
  if constexpr (FUSED) {
    if (!p.merge_inline) return;
    // ---- the query group's last CTA to finish merges its runs
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int old = atomicAdd(p.runs.ticket + (long long)b * gridDim.y + blockIdx.y, 1);
      *last_flag = old == (int)gridDim.x - 1 ? 1 : (old >= (int)gridDim.x ? -1 : 0);
    }
    __syncthreads();
    const int lf = *last_flag;
    if (lf < 0 && tid == 0) report(p.status, LCS_ERR_DEVICE_GUARD);   // ticket not zero at the start
    if (lf != 1) return;
    __threadfence();
    // the candidate buffers and the ring are idle now: the lists are staged from the first on
    uint64_t* stage = cand_s;
    int* run_off = reinterpret_cast<int*>(smem + ring_off + L::kRunOffR);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + ring_off + L::kHistR);
    const int stage_cap = (ring_off + L::kHistR - L::kCand) / 8;
#pragma unroll 1
    for (int qi = 0; qi < qn; ++qi)
      merge_query_topk<kThreads, 0, 11>(p.runs, qrow0 + qi, (n0 + qi + 1) >> mshift, k, stage, stage_cap, run_off,
                                        hist, p.out_idx, p.out_cnt, sel_all);
    if (tid == 0) {   // left at zero for the next call
      p.runs.ticket[(long long)b * gridDim.y + blockIdx.y] = 0;
      if (p.runs.gthr != nullptr)
        for (int qi = 0; qi < qn; ++qi) p.runs.gthr[qrow0 + qi] = 0ull;
    }
  }
}

// the merge kernel's shared memory: scratch, histogram, run offsets, then room for the lists
constexpr int kMergeHist = ((int)sizeof(SelScratch<256>) + 15) / 16 * 16;
constexpr int kMergeRunOff = kMergeHist + 2048 * 4;
constexpr int kMergeStage = kMergeRunOff + (kMaxRuns + 4) * 4;

// One CTA per query: the merge of the query's run lists (the selection phase on its own, or run
// lists too long for the scorer's shared memory).  grid: (max_new, num_seqs), block 256.
__global__ void __launch_bounds__(256) topk_merge_kernel(IndexParams p) {
  extern __shared__ __align__(16) uint8_t merge_smem[];
  const int b = blockIdx.y, i = blockIdx.x;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  if (i >= sp.qn) return;
  SelScratch<256>& sc = *reinterpret_cast<SelScratch<256>*>(merge_smem);
  uint32_t* hist = reinterpret_cast<uint32_t*>(merge_smem + kMergeHist);
  int* run_off = reinterpret_cast<int*>(merge_smem + kMergeRunOff);
  uint64_t* stage = reinterpret_cast<uint64_t*>(merge_smem + kMergeStage);
  const int t = sp.n0() + i;
  // (the stage holds the lists; the selection reads them with the lower bound, no candidate array)
  merge_query_topk<256, 0, 11>(p.runs, sp.q0 + i, (t + 1) / p.m, p.top_k, stage, p.runs.runs * p.runs.list_cap, run_off,
                               hist, p.out_idx, p.out_cnt, sc);
  if (threadIdx.x == 0 && p.runs.gthr != nullptr) p.runs.gthr[sp.q0 + i] = 0ull;   // left at zero
}

// ----------------------------------------------------------------------------------------------
// launcher
// ----------------------------------------------------------------------------------------------

namespace {

template <int HI, int QH>
size_t tc_smem_bytes(bool fused, int cap, int pages, int stages) {
  return stages == kStagesShallow ? TcSmem<QH, QH / HI, kStagesShallow>::bytes(fused, cap, pages)
                                  : TcSmem<QH, QH / HI, kStagesDeep>::bytes(fused, cap, pages);
}

size_t tc_smem_for(int heads, int qh, bool fused, int cap, int pages, int stages) {
  switch (heads * 100 + qh) {
    case 104: return tc_smem_bytes<1, 4>(fused, cap, pages, stages);
    case 204: return tc_smem_bytes<2, 4>(fused, cap, pages, stages);
    case 208: return tc_smem_bytes<2, 8>(fused, cap, pages, stages);
    case 404: return tc_smem_bytes<4, 4>(fused, cap, pages, stages);
    case 408: return tc_smem_bytes<4, 8>(fused, cap, pages, stages);
    case 416: return tc_smem_bytes<4, 16>(fused, cap, pages, stages);
    case 808: return tc_smem_bytes<8, 8>(fused, cap, pages, stages);
    case 816: return tc_smem_bytes<8, 16>(fused, cap, pages, stages);
    default: return 0;
  }
}

template <int HI, int QH>
size_t tc_stage_bytes(int cap, int stages) {
  return stages == kStagesShallow ? TcSmem<QH, QH / HI, kStagesShallow>::stage_bytes(cap)
                                  : TcSmem<QH, QH / HI, kStagesDeep>::stage_bytes(cap);
}

// bytes from the candidate buffers to the ring's histogram: the merge's staging room
size_t tc_stage_bytes_for(int heads, int qh, int cap, int stages) {
  switch (heads * 100 + qh) {
    case 104: return tc_stage_bytes<1, 4>(cap, stages);
    case 204: return tc_stage_bytes<2, 4>(cap, stages);
    case 208: return tc_stage_bytes<2, 8>(cap, stages);
    case 404: return tc_stage_bytes<4, 4>(cap, stages);
    case 408: return tc_stage_bytes<4, 8>(cap, stages);
    case 416: return tc_stage_bytes<4, 16>(cap, stages);
    case 808: return tc_stage_bytes<8, 8>(cap, stages);
    case 816: return tc_stage_bytes<8, 16>(cap, stages);
    default: return 0;
  }
}

template <int HI, int QH, bool FUSED, int ST>
cudaError_t launch_tc_st(const CUtensorMap& tmap, const CUtensorMap& tmap_t, const IndexParams& p,
                         const IndexTcPlan& plan, cudaStream_t st) {
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<HI, QH, FUSED, ST>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(index_tc_kernel<HI, QH, FUSED, ST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               100);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  dim3 grid(plan.runs, plan.groups, p.num_seqs);
  index_tc_kernel<HI, QH, FUSED, ST><<<grid, kThreads, plan.smem, st>>>(tmap, tmap_t, p, plan.tpc);
  return cudaGetLastError();
}

// the scores alone always take the deep ring (no candidate buffers to make room for)
template <int HI, int QH, bool FUSED>
cudaError_t launch_tc_t(const CUtensorMap& tmap, const CUtensorMap& tmap_t, const IndexParams& p,
                        const IndexTcPlan& plan, cudaStream_t st) {
  if constexpr (FUSED) {
    if (plan.stages == kStagesShallow) return launch_tc_st<HI, QH, true, kStagesShallow>(tmap, tmap_t, p, plan, st);
  }
  return launch_tc_st<HI, QH, FUSED, kStagesDeep>(tmap, tmap_t, p, plan, st);
}

template <bool FUSED>
cudaError_t launch_tc_switch(int heads, int qh, const CUtensorMap& tmap, const CUtensorMap& tmap_t, const IndexParams& p,
                             const IndexTcPlan& plan,
                             cudaStream_t st) {
  switch (heads * 100 + qh) {
    case 104: return launch_tc_t<1, 4, FUSED>(tmap, tmap_t, p, plan, st);
    case 204: return launch_tc_t<2, 4, FUSED>(tmap, tmap_t, p, plan, st);
    case 208: return launch_tc_t<2, 8, FUSED>(tmap, tmap_t, p, plan, st);
    case 404: return launch_tc_t<4, 4, FUSED>(tmap, tmap_t, p, plan, st);
    case 408: return launch_tc_t<4, 8, FUSED>(tmap, tmap_t, p, plan, st);
    case 416: return launch_tc_t<4, 16, FUSED>(tmap, tmap_t, p, plan, st);
    case 808: return launch_tc_t<8, 8, FUSED>(tmap, tmap_t, p, plan, st);
    case 816: return launch_tc_t<8, 16, FUSED>(tmap, tmap_t, p, plan, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Columns (query-heads) per 32-code block the tensor-core scorer uses, or 0 when it does not
// apply (rank other than 128, pages outside 8..128 entries, key codes not 32-byte or scales not
// 16-byte aligned).  Up to 4 queries per sequence: all of them in one CTA; longer query runs (k >
// 0, the fused top-k of a prefill chunk): groups of min(4, 16 / heads) queries.
int index_tc_qh(const IndexParams& p, int rank, int max_new, bool groups) {
  if (rank != 128 || p.paging.epb < 8 || p.paging.epb > 128 || (p.paging.epb & (p.paging.epb - 1))) return 0;
  if ((reinterpret_cast<uintptr_t>(p.k_fp4) & 31u) || (reinterpret_cast<uintptr_t>(p.k_scale) & 15u)) return 0;
  if (p.k_rows < p.paging.epb || p.k_rows > (1ll << 31)) return 0;
  if (p.heads != 1 && p.heads != 2 && p.heads != 4 && p.heads != 8) return 0;
  if (max_new < 1) return 0;
  if (max_new > 4) return groups ? std::min(4, 16 / p.heads) * p.heads : 0;
  const int need = max_new * p.heads;
  const int qh = need <= 4 ? 4 : (need <= 8 ? 8 : (need <= 16 ? 16 : 0));
  if (qh == 0 || qh / p.heads < max_new) return 0;
  return qh;
}

// The scorer's grid and shared memory; with k > 0 the fused top-k (applies = 0 when the
// candidate buffers or the merge bitmap do not fit).  The fused top-k takes the shallow ring when
// the last CTA can stage every run's list in it (its candidate buffers then have room for about
// 4 KB more keys each), else the deep ring.
IndexTcPlan plan_index_tc(const IndexParams& p, int rank, int max_new, int max_entries, int num_seqs, int sms, int k) {
  IndexTcPlan plan{};
  const bool fused = k > 0;
  plan.qh = index_tc_qh(p, rank, max_new, fused);
  if (plan.qh == 0) return plan;
  const int qps = plan.qh / p.heads;
  plan.groups = (max_new + qps - 1) / qps;
  if (plan.groups > 65535) return plan;
  const int tiles = std::max(1, (max_entries + kTile - 1) / kTile);
  const int epb = p.paging.epb;
  int tpc_cap = kMaxPages * epb / kTile;                       // a run spans at most kMaxPages pages
  // a sequence has at most kMaxRuns runs, and no more than the merge kernel can stage the lists of
  const int runs_max = fused ? std::max(1, std::min(kMaxRuns, (227 * 1024 - kMergeStage) / (8 * k))) : kMaxRuns;
  const int tpc_min = (tiles + runs_max - 1) / runs_max;   // fewer runs: longer ones
  tpc_cap = std::max(tpc_cap, tpc_min);
  if (tpc_cap * kTile / epb > 4 * kMaxPages) return plan;
  // resident CTAs per SM: tensor memory and registers (16 query-head columns take 168 registers a
  // thread: one CTA), then shared memory below
  const int occ_tmem = std::min(512 / (int)tmem_cols_for(4 * plan.qh), plan.qh >= 16 ? 1 : 2);
  // a compaction keeps at most k + k/8 keys and leaves room for the epilogue's next two tiles
  const int cap_min = fused ? (k + (k >> 3) + 2 * kTile + 15) / 16 * 16 : 0;
  auto attempt = [&](int stages) {
    IndexTcPlan pl = plan;
    pl.stages = stages;
    // two resident CTAs per SM when their shared memory allows it, else one
    for (int occ = std::min(2, occ_tmem); occ >= 1; --occ) {
      int runs = std::max(1, (sms * occ) / std::max(1, num_seqs * pl.groups));   // about one wave
      int tpc = std::max(tpc_min, std::min(tpc_cap, (tiles + runs - 1) / runs));
      runs = (tiles + tpc - 1) / tpc;
      const int pages = tpc * kTile / epb + 1;
      const long long budget = std::min<long long>((long long)(228 * 1024 / occ) - 1024, 227 * 1024);
      const long long base = (long long)tc_smem_for(p.heads, pl.qh, fused, 0, pages, stages);
      if ((long long)tc_smem_for(p.heads, pl.qh, fused, cap_min, pages, stages) > budget) continue;
      int cap = cap_min;
      if (fused) {   // more candidate room while it fits, up to a whole run's entries: fewer compactions
        const int fit = (int)((budget - base) / (8ll * qps)) / (2 * kTile) * (2 * kTile);
        cap = std::max(cap_min, std::min(fit, (tpc + 2) * kTile));
        // (the ring after the buffers is 1024-aligned: give back room until the whole fits)
        while (cap > cap_min && (long long)tc_smem_for(p.heads, pl.qh, fused, cap, pages, stages) > budget)
          cap = std::max(cap_min, cap - 2 * kTile);
      }
      pl.runs = runs;
      pl.tpc = tpc;
      pl.cap = cap;
      pl.smem = tc_smem_for(p.heads, pl.qh, fused, cap, pages, stages);
      pl.applies = 1;
      break;
    }
    if (!pl.applies) return pl;
    // the last CTA merges in place when the runs' lists fit its idle ring; a run's bitmap and word
    // prefixes fit it in any case (tpc * 128 entries: at most 8 bits of ring per entry)
    const size_t stage_bytes = tc_stage_bytes_for(p.heads, pl.qh, pl.cap, stages);
    const size_t bitmap_bytes = stages == kStagesShallow ? (size_t)TcSmem<16, 4, kStagesShallow>::kHistR
                                                         : (size_t)TcSmem<16, 4, kStagesDeep>::kHistR;
    // lists with slack (k/4, else k/8) when they fit the staging room, else exact ones
    pl.list_cap = k;
    for (const int lc : {topk_list_cap(k), k + (k >> 3)})
      if (fused && pl.list_cap == k && (size_t)pl.runs * lc * 8 <= stage_bytes) pl.list_cap = lc;
    pl.merge_inline = fused && (size_t)pl.runs * pl.list_cap * 8 <= stage_bytes;
    pl.merge_smem = (size_t)kMergeStage + (size_t)pl.runs * pl.list_cap * 8;
    if (fused && (size_t)pl.tpc * kTile / 32 * 8 > bitmap_bytes) pl.applies = 0;
    if (fused && !pl.merge_inline && pl.merge_smem > 227 * 1024) pl.applies = 0;
    return pl;
  };
  if (fused) {
    const IndexTcPlan shallow = attempt(kStagesShallow);
    if (shallow.applies && shallow.merge_inline) return shallow;
  }
  return attempt(kStagesDeep);
}

cudaError_t launch_index_tc(const IndexParams& p, const IndexTcPlan& plan, cudaStream_t st) {
  if (!plan.applies) return cudaErrorInvalidValue;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // codes as [rows][64] bytes (two 4-bit codes each); a box of one page lands as rows of 64 bytes
  // with the 64-byte swizzle, the packed operand form of kind::mxf4
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {64u, (cuuint64_t)p.k_rows};
  const cuuint64_t gstride[1] = {64u};
  const cuuint32_t box[2] = {64u, (cuuint32_t)p.paging.epb};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.k_fp4), gdim, gstride, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // the same codes in boxes of a whole tile (128 rows), for tiles whose pages are consecutive
  CUtensorMap tmap_t = tmap;
  if (p.k_rows >= kTile) {
    const cuuint32_t box_t[2] = {64u, (cuuint32_t)kTile};
    r = enc(&tmap_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.k_fp4), gdim, gstride, box_t, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  if (p.scores_out != nullptr) return launch_tc_switch<false>(p.heads, plan.qh, tmap, tmap_t, p, plan, st);
  return launch_tc_switch<true>(p.heads, plan.qh, tmap, tmap_t, p, plan, st);
}

cudaError_t launch_topk_merge(const IndexParams& p, const IndexTcPlan& plan, int max_new, cudaStream_t st) {
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    return cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (ea != cudaSuccess) return ea;
  dim3 grid(max_new, p.num_seqs);
  if (grid.x == 0) return cudaSuccess;
  topk_merge_kernel<<<grid, 256, plan.merge_smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lcsa
