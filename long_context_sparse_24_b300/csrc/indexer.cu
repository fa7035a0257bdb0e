// Lightning indexer scores and causal top-k selection.
//
// Defined by: m.x-techcon.com/article/133366, section 2, CSA step 2 (a lightweight low-rank
// indexer scores every compressed entry; each query keeps the top-k entries, k = 1024 Pro /
// 512 Flash) and section 4 "FP4量化感知训练" (the indexer's QK path is FP4; FP4 -> FP8 is
// lossless because FP8 has two more exponent bits).  digipub.cc "DeepSeek V4來了", section
// "把賬算在注意力機制上": top-k sparse attention continuing V3.2's DSA.
//
// score(i, j) = sum_h w[i,h] * phi( sum_blk 2^(eq+ek) * sum_{c in blk} q[c] * k[c] )
//
// Scores: E2M1 codes are widened to E4M3 in registers (a lossless re-encoding) and multiplied
// with the warp-level m16n8k32 E4M3 MMA, one MMA per 32-element block so the block scales can
// be applied afterwards in fp32.  Every partial sum of one block is an integer multiple of 1/4
// below 2^11, so the MMA result is exact; the scaled sums across blocks and heads stay exact
// in fp32 for the documented exponent ranges.  Row / column roles: A = 16 entries x 32 codes,
// B = 32 codes x 8 (query, head) columns.  Thread t of a quad loads 32-bit word t of a block
// (codes 8t..8t+7) for both operands and widens it into the two registers that hold MMA
// k-slots 4t..4t+3 and 16+4t..16+4t+3: both operands use the same code -> k-slot map, so the
// MMA computes the block's dot product.
//
// Top-k: scores are mapped to order-preserving 32-bit keys; a per-query radix select (three
// digit passes of 11/11/10 bits) finds the k-th largest key T and how many keys equal to T are
// taken; an ordered block-wide compaction then emits the selected j in ascending order, taking
// keys equal to T lowest-j first.
#include "kernels.cuh"

namespace lcsa {



// E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 as E4M3 bytes.
constexpr uint32_t kLut0 = 0x3C383000u;
constexpr uint32_t kLut1 = 0x4C484440u;

// prmt.b32 in its default mode: result byte n is picked by selector nibble n (bits 0-2 index the
// eight bytes of {a, b}; bit 3 set replicates the picked byte's top bit over the result byte).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// 8 E2M1 codes (one 32-bit word, code n in bits 4n..4n+3) -> 8 E4M3 codes:
// lo = codes 0..3 (bytes 0..3), hi = codes 4..7.  Magnitudes come from the 8-entry table,
// signs from the code's top bit.
__device__ __forceinline__ void widen_e2m1(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t ws = w << 4;                 // byte k of ws carries code 2k's sign as its top bit
  const uint32_t mlo = prmt(kLut0, kLut1, w & 0x7777u);
  const uint32_t mhi = prmt(kLut0, kLut1, (w >> 16) & 0x7777u);
  const uint32_t slo = prmt(ws, w, 0xD9C8u);  // codes 0,1,2,3 <- top bits of ws.b0, w.b0, ws.b1, w.b1
  const uint32_t shi = prmt(ws, w, 0xFBEAu);  // codes 4,5,6,7 <- top bits of ws.b2, w.b2, ws.b3, w.b3
  lo = mlo | (slo & 0x80808080u);
  hi = mhi | (shi & 0x80808080u);
}

template <int NT, int RB>
__global__ void __launch_bounds__(256) index_score_kernel(IndexParams p) {
  constexpr int TPW = 8;                       // 16-entry tiles per warp
  constexpr int CHUNK = 8 * TPW * 16;          // entries per CTA
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int Hi = p.heads;
  const int QPT = 8 / Hi;                      // queries per n8 tile
  const int QG = QPT * NT;                     // queries per CTA
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int qbase = blockIdx.y * QG;
  if (qbase >= sp.qn) return;
  const int qcount = min(QG, sp.qn - qbase);
  const int n0 = sp.n0();
  const int nmax = (n0 + qbase + qcount) / p.m;     // N(t) of the last query of the group
  const int chunk0 = blockIdx.x * CHUNK;
  if (chunk0 >= nmax) return;
  constexpr int rh = RB * 16;                  // bytes per FP4 row (r/2)

  // ---- query operands (B) and per-column scales / weights
  uint32_t bq[NT][RB][2];
  float qsc[NT][RB][2];
  float hw[NT][2];
  int colq[NT][2];                             // query index (within group) of the thread's C columns
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi_b = nt * QPT + g / Hi, h_b = g % Hi;
    const bool vb = qi_b < qcount;
    const long long qrow = (long long)(sp.q0 + qbase + qi_b) * Hi + h_b;
#pragma unroll
    for (int blk = 0; blk < RB; ++blk) {
      uint32_t w = vb ? *reinterpret_cast<const uint32_t*>(p.q_fp4 + qrow * rh + blk * 16 + t4 * 4) : 0u;
      widen_e2m1(w, bq[nt][blk][0], bq[nt][blk][1]);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = 2 * t4 + c;
      const int qi = nt * QPT + col / Hi, h = col % Hi;
      const bool v = qi < qcount;
      colq[nt][c] = v ? qi : -1;
      const long long qr = (long long)(sp.q0 + qbase + (v ? qi : 0)) * Hi + h;
      hw[nt][c] = v ? (p.head_w ? p.head_w[qr] : 1.0f) : 0.0f;
#pragma unroll
      for (int blk = 0; blk < RB; ++blk) qsc[nt][blk][c] = v ? ue8m0_to_f32(p.q_scale[qr * RB + blk]) : 0.0f;
    }
  }

  for (int it = 0; it < TPW; ++it) {
    const int e0 = chunk0 + (it * 8 + warp) * 16;
    if (e0 >= nmax) break;
    // ---- key operands (A): rows g and g+8 of the tile
    uint32_t a[RB][4];
    float ksc[2][RB];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int j = e0 + g + 8 * half;
      long long row = -1;
      if (j < nmax) {
        row = entry_row(p.paging, b, j, p.k_rows);
        if (row < 0) report(p.status, LCS_ERR_DEVICE_GUARD);
      }
      uint32_t sc = 0x7F7F7F7Fu;
      if (row >= 0) {
        if (RB == 4) sc = *reinterpret_cast<const uint32_t*>(p.k_scale + row * RB);
        else sc = *reinterpret_cast<const uint16_t*>(p.k_scale + row * RB);
      }
#pragma unroll
      for (int blk = 0; blk < RB; ++blk) {
        uint32_t w = row >= 0 ? *reinterpret_cast<const uint32_t*>(p.k_fp4 + row * rh + blk * 16 + t4 * 4) : 0u;
        uint32_t lo, hi;
        widen_e2m1(w, lo, hi);
        // A registers: a0 (row g, k 0..3 of this thread), a1 (row g+8), a2 (row g, k 16..19), a3 (row g+8)
        a[blk][half] = lo;
        a[blk][2 + half] = hi;
        ksc[half][blk] = ue8m0_to_f32((sc >> (8 * blk)) & 0xFF);
      }
    }
    // ---- MMAs, one per block, scaled and accumulated in fp32
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int blk = 0; blk < RB; ++blk) {
        float d[4];
        mma_e4m3_zero(d, a[blk][0], a[blk][1], a[blk][2], a[blk][3], bq[nt][blk][0], bq[nt][blk][1]);
        acc[0] = fmaf(d[0], ksc[0][blk] * qsc[nt][blk][0], acc[0]);
        acc[1] = fmaf(d[1], ksc[0][blk] * qsc[nt][blk][1], acc[1]);
        acc[2] = fmaf(d[2], ksc[1][blk] * qsc[nt][blk][0], acc[2]);
        acc[3] = fmaf(d[3], ksc[1][blk] * qsc[nt][blk][1], acc[3]);
      }
      if (p.relu) {
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = fmaxf(acc[c], 0.0f);
      }
      // ---- head combination and write-out
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int j = e0 + g + 8 * half;
        float s0 = acc[2 * half] * hw[nt][0];
        float s1 = acc[2 * half + 1] * hw[nt][1];
        if (Hi == 1) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int qi = colq[nt][c];
            const float s = c == 0 ? s0 : s1;
            if (qi >= 0 && j < (n0 + qbase + qi + 1) / p.m) {
              const long long o = (long long)(sp.q0 + qbase + qi) * p.ld + j;
              if (p.scores_out) p.scores_out[o] = s;
              else p.keys_out[o] = score_key(s);
            }
          }
        } else {
          float s = s0 + s1;
          if (Hi >= 4) s += __shfl_xor_sync(0xffffffffu, s, 1);
          if (Hi >= 8) s += __shfl_xor_sync(0xffffffffu, s, 2);
          const int lead = Hi == 2 ? 1 : (Hi == 4 ? 2 : 4);
          const int qi = colq[nt][0];
          if ((t4 % lead) == 0 && qi >= 0 && j < (n0 + qbase + qi + 1) / p.m) {
            const long long o = (long long)(sp.q0 + qbase + qi) * p.ld + j;
            if (p.scores_out) p.scores_out[o] = s;
            else p.keys_out[o] = score_key(s);
          }
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------------------------
// top-k selection
// ----------------------------------------------------------------------------------------------

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kHistBins = 2048;
constexpr int kSelCacheKeys = 40960;   // keys kept in shared memory when N fits (160 KB)

struct SelectShared {
  uint32_t hist[kHistBins];
  int warp_tot[2][kSelWarps];
  int found_bin;
  int found_above;
};

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix, total in *tot.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    int tw = warp_tot[w];
    before += (w < warp) ? tw : 0;
    all += tw;
  }
  __syncthreads();
  *tot = all;
  return before + x - v;
}

// grid: (max_new, num_seqs); block kSelThreads; dynamic smem: SelectShared + cache.
__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(const uint32_t* keys, long long ld,
                                                                 const int32_t* cu_new, const int32_t* seq_len,
                                                                 int m, int k, int32_t* out_idx, int32_t* out_cnt,
                                                                 int use_cache) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectShared& sh = *reinterpret_cast<SelectShared*>(smem_raw);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem_raw + sizeof(SelectShared));
  const int b = blockIdx.y, i = blockIdx.x, tid = threadIdx.x;
  const SeqSpan sp = seq_span(cu_new, seq_len, b);
  if (i >= sp.qn) return;
  const int t = sp.n0() + i;
  const int N = (t + 1) / m;
  const long long q = (long long)sp.q0 + i;
  int32_t* out = out_idx + q * k;
  if (N <= k) {
    for (int j = tid; j < k; j += kSelThreads) out[j] = j < N ? j : -1;
    if (tid == 0) out_cnt[q] = N;
    return;
  }
  const uint32_t* src = keys + q * ld;
  if (use_cache && N <= kSelCacheKeys) {
    for (int j = tid; j < N; j += kSelThreads) cache[j] = src[j];
    src = cache;
  }
  __syncthreads();

  uint32_t prefix = 0;
  int remaining = k;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh_ = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    const int hi_shift = sh_ + widths[pass];   // bits at and above this must match the prefix
    for (int d = tid; d < kHistBins; d += kSelThreads) sh.hist[d] = 0;
    __syncthreads();
    for (int j = tid; j < N; j += kSelThreads) {
      const uint32_t u = src[j];
      const bool match = hi_shift >= 32 ? true : ((u >> hi_shift) == (prefix >> hi_shift));
      if (match) atomicAdd(&sh.hist[(u >> sh_) & dmask], 1u);
    }
    __syncthreads();
    // thread `tid` owns bins top-down: d = 2047 - 4*tid - r
    int cnt[4];
    int local = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      cnt[r] = (int)sh.hist[kHistBins - 1 - 4 * tid - r];
      local += cnt[r];
    }
    int tot;
    int running = block_excl_scan(local, sh.warp_tot[0], &tot);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (running < remaining && running + cnt[r] >= remaining) {
        sh.found_bin = kHistBins - 1 - 4 * tid - r;
        sh.found_above = running;
      }
      running += cnt[r];
    }
    __syncthreads();
    prefix |= (uint32_t)sh.found_bin << sh_;
    remaining -= sh.found_above;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int need_eq = remaining;   // keys equal to T to take, lowest j first

  int base = 0, eq_seen = 0;
  const unsigned lt_mask = (1u << (tid & 31)) - 1u;
  for (int j0 = 0; j0 < N; j0 += kSelThreads) {
    const int j = j0 + tid;
    const uint32_t u = j < N ? src[j] : 0u;
    const bool gt = j < N && u > T;
    const bool eq = j < N && u == T;
    int eq_tot;
    const int eq_rank = eq_seen + block_excl_scan(eq ? 1 : 0, sh.warp_tot[0], &eq_tot);
    const bool sel = gt || (eq && eq_rank < need_eq);
    int sel_tot;
    const int pos = base + block_excl_scan(sel ? 1 : 0, sh.warp_tot[1], &sel_tot);
    if (sel && pos < k) out[pos] = j;
    base += sel_tot;
    eq_seen += eq_tot;
    (void)lt_mask;
  }
  if (tid == 0) out_cnt[q] = k;
}

// ----------------------------------------------------------------------------------------------
// launchers
// ----------------------------------------------------------------------------------------------

cudaError_t launch_index_scores(const IndexParams& p, int rank, int max_new, int max_entries, cudaStream_t st) {
  const bool prefill = max_new > 2;
  const int NT = prefill ? 4 : 1;
  const int QG = (8 / p.heads) * NT;
  constexpr int CHUNK = 8 * 8 * 16;
  dim3 grid((max_entries + CHUNK - 1) / CHUNK, (max_new + QG - 1) / QG, p.num_seqs);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  if (rank == 128) {
    if (prefill) index_score_kernel<4, 4><<<grid, 256, 0, st>>>(p);
    else index_score_kernel<1, 4><<<grid, 256, 0, st>>>(p);
  } else {
    if (prefill) index_score_kernel<4, 2><<<grid, 256, 0, st>>>(p);
    else index_score_kernel<1, 2><<<grid, 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

size_t select_smem_bytes(bool cache) {
  return sizeof(SelectShared) + (cache ? (size_t)kSelCacheKeys * 4 : 0);
}

cudaError_t launch_topk_select(const uint32_t* keys, long long ld, const int32_t* cu_new, const int32_t* seq_len,
                               int num_seqs, int max_new, int m, int k, int max_entries, int32_t* out_idx,
                               int32_t* out_cnt, cudaStream_t st) {
  const bool cache = max_entries <= kSelCacheKeys;
  const size_t smem = select_smem_bytes(cache);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)select_smem_bytes(true));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(max_new, num_seqs);
  if (grid.x == 0) return cudaSuccess;
  topk_select_kernel<<<grid, kSelThreads, smem, st>>>(keys, ld, cu_new, seq_len, m, k, out_idx, out_cnt,
                                                       cache ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace lcsa
