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
  extern __shared__ uint32_t hist_s[];         // [QG][kTopkHistBins] when p.hist != null
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
  const bool with_hist = p.hist != nullptr;
  if (with_hist) {
    for (int i = threadIdx.x; i < QG * kTopkHistBins; i += blockDim.x) hist_s[i] = 0;
    __syncthreads();
  }

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
              if (p.scores_out) {
                p.scores_out[o] = s;
              } else {
                const uint32_t key = score_key(s);
                p.keys_out[o] = key;
                if (with_hist) atomicAdd(&hist_s[qi * kTopkHistBins + (key >> 21)], 1u);
              }
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
            if (p.scores_out) {
              p.scores_out[o] = s;
            } else {
              const uint32_t key = score_key(s);
              p.keys_out[o] = key;
              if (with_hist) atomicAdd(&hist_s[qi * kTopkHistBins + (key >> 21)], 1u);
            }
          }
        }
      }
    }
  }
  if (with_hist) {
    __syncthreads();
    for (int i = threadIdx.x; i < qcount * kTopkHistBins; i += blockDim.x) {
      const uint32_t c = hist_s[i];
      if (c) atomicAdd(&p.hist[(long long)(sp.q0 + qbase + i / kTopkHistBins) * kTopkHistBins + i % kTopkHistBins], c);
    }
  }
}

// ----------------------------------------------------------------------------------------------
// top-k selection
// ----------------------------------------------------------------------------------------------

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kHistBins = kTopkHistBins;
constexpr int kKPT = 16;                          // keys per thread per chunk
constexpr int kChunkKeys = kSelThreads * kKPT;    // 8192
constexpr int kCandCap = 8192;                    // (key, j) pairs kept in shared memory

struct SelectShared {
  uint32_t hist[kHistBins];
  int warp_tot[2][kSelWarps];
  int found_bin;
  int found_above;
  uint32_t cand_key[kCandCap];
  int32_t cand_j[kCandCap];
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

// Highest bin d with (count of bins above d) < remaining <= (count of bins >= d).  Thread tid
// owns bins 2047-4*tid .. 2044-4*tid.  Result in sh.found_bin / sh.found_above.
__device__ __forceinline__ void find_bin(SelectShared& sh, int remaining) {
  const int tid = threadIdx.x;
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
}

// Exact radix select over `n` keys read through `key_at`; bits above `start_shift + width` of
// every counted key must equal `prefix`.  Returns the k-th key; *need_eq = ties to take.
template <typename KeyAt>
__device__ uint32_t radix_select(SelectShared& sh, int n, KeyAt key_at, uint32_t prefix, int remaining, int npass,
                                 const int* shifts, const int* widths, int* need_eq) {
  for (int pass = 0; pass < npass; ++pass) {
    const int sh_ = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    const int hi_shift = sh_ + widths[pass];
    for (int d = threadIdx.x; d < kHistBins; d += kSelThreads) sh.hist[d] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kSelThreads) {
      const uint32_t u = key_at(i);
      const bool match = hi_shift >= 32 ? true : ((u >> hi_shift) == (prefix >> hi_shift));
      if (match) atomicAdd(&sh.hist[(u >> sh_) & dmask], 1u);
    }
    __syncthreads();
    find_bin(sh, remaining);
    prefix |= (uint32_t)sh.found_bin << sh_;
    remaining -= sh.found_above;
    __syncthreads();
  }
  *need_eq = remaining;
  return prefix;
}

// Ordered emission: out[pos] = j for every selected key, j ascending.
template <typename KeyAt, typename IdxAt>
__device__ void emit_selected(SelectShared& sh, int n, KeyAt key_at, IdxAt idx_at, uint32_t T, int need_eq,
                              int32_t* out, int k) {
  int base = 0, eq_seen = 0;
  for (int i0 = 0; i0 < n; i0 += kSelThreads) {
    const int i = i0 + threadIdx.x;
    const uint32_t u = i < n ? key_at(i) : 0u;
    const bool gt = i < n && u > T;
    const bool eq = i < n && u == T;
    int eq_tot;
    const int eq_rank = eq_seen + block_excl_scan(eq ? 1 : 0, sh.warp_tot[0], &eq_tot);
    const bool sel = gt || (eq && eq_rank < need_eq);
    int sel_tot;
    const int pos = base + block_excl_scan(sel ? 1 : 0, sh.warp_tot[1], &sel_tot);
    if (sel && pos < k) out[pos] = idx_at(i);
    base += sel_tot;
    eq_seen += eq_tot;
  }
}

// grid: (max_new, num_seqs); block kSelThreads; dynamic smem sizeof(SelectShared).
// hist: the per-query histogram of key >> 21 built by the score kernel.
__global__ void __launch_bounds__(kSelThreads, 2) topk_select_kernel(const uint32_t* keys, const uint32_t* hist,
                                                                 long long ld, const int32_t* cu_new,
                                                                 const int32_t* seq_len, int m, int k,
                                                                 int32_t* out_idx, int32_t* out_cnt) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectShared& sh = *reinterpret_cast<SelectShared*>(smem_raw);
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

  // 1. bin of the k-th largest key from the score kernel's histogram
  for (int d = tid; d < kHistBins; d += kSelThreads) sh.hist[d] = hist[q * kHistBins + d];
  __syncthreads();
  find_bin(sh, k);
  const uint32_t b1 = (uint32_t)sh.found_bin;
  const int above1 = sh.found_above;
  __syncthreads();

  // 2. one ordered pass: keep (key, j) of every key in bin b1 or above, j ascending
  int ncand = 0;
  bool overflow = false;
  for (int c0 = 0; c0 < N; c0 += kChunkKeys) {
    const int j0 = c0 + tid * kKPT;
    // the next chunk toward L2 while this one is scanned (long prefill rows are not L2-resident)
    if (j0 + kChunkKeys + kKPT <= N)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(src + j0 + kChunkKeys) : "memory");
    uint32_t u[kKPT];
    if (j0 + kKPT <= N) {
      const uint4* v = reinterpret_cast<const uint4*>(src + j0);
#pragma unroll
      for (int w = 0; w < kKPT / 4; ++w) {
        const uint4 x = v[w];
        u[4 * w] = x.x; u[4 * w + 1] = x.y; u[4 * w + 2] = x.z; u[4 * w + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < kKPT; ++e) u[e] = (j0 + e < N) ? src[j0 + e] : 0u;
    }
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < kKPT; ++e) cnt += (j0 + e < N && (u[e] >> 21) >= b1) ? 1 : 0;
    int tot;
    int pos = ncand + block_excl_scan(cnt, sh.warp_tot[0], &tot);
    if (ncand + tot > kCandCap) {   // uniform: tot is the block total
      overflow = true;
      break;
    }
#pragma unroll
    for (int e = 0; e < kKPT; ++e) {
      if (j0 + e < N && (u[e] >> 21) >= b1) {
        sh.cand_key[pos] = u[e];
        sh.cand_j[pos] = j0 + e;
        ++pos;
      }
    }
    ncand += tot;
  }
  __syncthreads();

  int need_eq;
  if (!overflow) {
    // 3. resolve the k-th key inside bin b1 (low 21 bits) among the kept keys
    const int shifts[2] = {10, 0};
    const int widths[2] = {11, 10};
    const uint32_t T = radix_select(sh, ncand, [&](int x) { return sh.cand_key[x]; }, b1 << 21, k - above1, 2,
                                    shifts, widths, &need_eq);
    // 4. ordered emission from the kept keys
    emit_selected(sh, ncand, [&](int x) { return sh.cand_key[x]; }, [&](int x) { return sh.cand_j[x]; }, T,
                  need_eq, out, k);
  } else {
    // degenerate distributions (very many keys near the k-th): full radix select over all keys
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    const uint32_t T = radix_select(sh, N, [&](int x) { return src[x]; }, 0u, k, 3, shifts, widths, &need_eq);
    emit_selected(sh, N, [&](int x) { return src[x]; }, [&](int x) { return x; }, T, need_eq, out, k);
  }
  if (tid == 0) out_cnt[q] = k;
}

// ----------------------------------------------------------------------------------------------
// launchers
// ----------------------------------------------------------------------------------------------

cudaError_t launch_index_scores(const IndexParams& p, int rank, int max_new, int max_entries, cudaStream_t st) {
  // queries per CTA = (8 / heads) * NT, kept at 8 or fewer so the CTA's histogram fits in 64 KB
  const bool prefill = max_new > 2;
  const int NT = prefill ? (p.heads >= 4 ? 4 : p.heads) : 1;
  const int QG = (8 / p.heads) * NT;
  constexpr int CHUNK = 8 * 8 * 16;
  dim3 grid((max_entries + CHUNK - 1) / CHUNK, (max_new + QG - 1) / QG, p.num_seqs);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  const size_t smem = p.hist ? (size_t)QG * kTopkHistBins * 4 : 0;
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    const int mx = 8 * kTopkHistBins * 4;
    cudaError_t e = cudaSuccess;
    for (auto fn : {index_score_kernel<4, 4>, index_score_kernel<2, 4>, index_score_kernel<1, 4>,
                    index_score_kernel<4, 2>, index_score_kernel<2, 2>, index_score_kernel<1, 2>})
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  if (rank == 128) {
    if (NT == 4) index_score_kernel<4, 4><<<grid, 256, smem, st>>>(p);
    else if (NT == 2) index_score_kernel<2, 4><<<grid, 256, smem, st>>>(p);
    else index_score_kernel<1, 4><<<grid, 256, smem, st>>>(p);
  } else {
    if (NT == 4) index_score_kernel<4, 2><<<grid, 256, smem, st>>>(p);
    else if (NT == 2) index_score_kernel<2, 2><<<grid, 256, smem, st>>>(p);
    else index_score_kernel<1, 2><<<grid, 256, smem, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_topk_select(const uint32_t* keys, const uint32_t* hist, long long ld, const int32_t* cu_new,
                               const int32_t* seq_len, int num_seqs, int max_new, int m, int k, int32_t* out_idx,
                               int32_t* out_cnt, cudaStream_t st) {
  const size_t smem = sizeof(SelectShared);
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [smem] {
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    // two CTAs per SM for long query runs (prefill): ask for the whole carveout as shared memory
    if (e == cudaSuccess) e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  dim3 grid(max_new, num_seqs);
  if (grid.x == 0) return cudaSuccess;
  topk_select_kernel<<<grid, kSelThreads, smem, st>>>(keys, hist, ld, cu_new, seq_len, m, k, out_idx, out_cnt);
  return cudaGetLastError();
}

}  // namespace lcsa
