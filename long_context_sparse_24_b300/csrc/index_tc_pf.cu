// Lightning-indexer scores on the tcgen05 tensor cores for long runs of queries per sequence
// (prefill chunks).
//
// Defined by: m.x-techcon.com/article/133366, section 2, CSA step 2 (a low-rank indexer scores
// every compressed entry, each query keeps its top-k) and section 4 "FP4量化感知训练" (the
// indexer's QK path runs in FP4).  Same arithmetic as the decode scorer in index_tc.cu:
//   score(q, j) = sum_h w[q,h] * phi( sum_blk 2^(eq[q,h,blk] + ek[j,blk]) * dot_blk(q_h, k_j) ).
//
// Work unit: one group of QPS consecutive queries of a sequence against a run of 128-entry
// tiles of that sequence (grid = runs x query groups x sequences).  The CTA is warp-specialised
// like the decode scorer -- two producer warps stream the tiles' E2M1 codes through TMA (the
// "16 x U4 in 16 bytes" form, 128-byte swizzle, i.e. the K-major E2M1 operand of kind::f8f6f4)
// plus their block scales through cp.async, one thread issues the MMAs -- but B holds the whole
// query group: N = 4 * HI * QPS rows, row (q, h, blk) = query q's head-h codes inside 32-code
// block blk and zeros elsewhere, so the four K = 32 MMAs of a tile leave every block's exact
// partial dot product in its own column (multiples of 1/4 below 2^11, exact in fp32), one
// query's 4*HI columns adjacent and the four blocks of a head adjacent.  Sixteen epilogue warps
// (four per TMEM lane quadrant, each a quarter of the group's queries) read a tile's columns,
// hand the accumulator back at once, and apply block scales and head weights in fp32, two
// blocks per packed f32x2 instruction.  The keys (order-preserving uint32 of the score) go to
// the caller's [T][ld] buffer and into a per-query 2048-bin shared-memory histogram of
// key >> 21 that the top-k selection starts from.
#include "kernels.cuh"
#include "sm100.cuh"

namespace lcsa {

namespace {

constexpr int kTile = 128;           // entries per MMA tile (M)
constexpr int kStages = 3;           // shared-memory ring depth
constexpr int kMaxPages = 1024;      // block-table entries one run may span
constexpr int kRowBytes = 128;       // shared-memory bytes of one entry's 128 codes (16U4 in 16 B)
constexpr int kPackedRowBytes = 64;  // global bytes of the same codes
constexpr int kATileBytes = kTile * kRowBytes;
constexpr int kEpiWarps = 16;        // four per TMEM lane quadrant, a quarter of the queries each
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kProdWarps = 2;
constexpr int kScaleSlots = 2 * kStages;
constexpr int kThreads = kEpiThreads + 32 * kProdWarps + 32;

template <int HI, int QPS>
struct PfSmem {
  static constexpr int N = 4 * HI * QPS;                        // MMA N
  static constexpr int kAcc = (512 / N) > 4 ? 4 : (512 / N);    // tensor-memory accumulators
  static constexpr int kCols = kAcc * N;                        // 256 or 512 (power of two)
  static constexpr int kA = 0;                                  // kStages x 16 KB, 1024-aligned
  static constexpr int kB = kA + kStages * kATileBytes;         // N x 128 B
  static constexpr int kScale = kB + N * kRowBytes;             // kScaleSlots x 128 x 4 B
  static constexpr int kQw = kScale + kScaleSlots * kTile * 4;  // f32 [QPS][HI][4] qscale * w
  static constexpr int kQs = kQw + QPS * 4 * HI * 4;            // f32 [QPS][HI][4] qscale
  static constexpr int kHw = kQs + QPS * HI * 4 * 4;            // f32 [QPS][HI] w
  static constexpr int kPages = kHw + QPS * HI * 4;             // int [kMaxPages]
  static constexpr int kBar = kPages + kMaxPages * 4;           // full/empty[kStages], accf/acce[kAcc]
  static constexpr int kMisc = kBar + (2 * kStages + 2 * kAcc) * 8;
  static constexpr int kHist = kMisc + 16;                      // u32 [QPS][2048]
  static constexpr int kBytes = kHist + QPS * kTopkHistBins * 4 + 1024;
  static_assert(kCols == 256 || kCols == 512, "TMEM allocation must be a power of two >= 32");
  static_assert(kB % 1024 == 0, "B operand must stay 1024-aligned for the 128-byte swizzle");
};

}  // namespace

// packed pairs of fp32 (two IEEE operations per instruction)
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_sum(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <int HI, int QPS>
__global__ void __launch_bounds__(kThreads, 1) index_tc_pf_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                              IndexParams p, int tiles_per_cta) {
  using L = PfSmem<HI, QPS>;
  constexpr int N = L::N;
  constexpr int kAcc = L::kAcc;
  constexpr int V = 4 * HI;                                  // columns per query
  constexpr uint32_t kIdesc = idesc_f8f6f4(5, 5, kTile, N);  // E2M1 x E2M1 -> f32, M = 128
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int g0 = blockIdx.y * QPS;                // first query of the group (within the sequence)
  const int qn = min(sp.qn - g0, QPS);
  if (qn <= 0) return;
  const int n0 = sp.n0() + g0;                    // position of the group's first query
  const long long q0 = (long long)sp.q0 + g0;     // its row in the batch
  const int mshift = 31 - __clz(p.m);
  const int nmax = (n0 + qn) >> mshift;           // visible entries of the group's last query
  const int t_begin = blockIdx.x * tiles_per_cta;
  const int t_end = min((nmax + kTile - 1) / kTile, t_begin + tiles_per_cta);
  if (t_begin >= t_end) return;
  const int nt = t_end - t_begin;
  const bool with_hist = p.hist != nullptr;
  const int epb = p.paging.epb;
  const int eshift = 31 - __clz(epb);
  const int page0 = (t_begin * kTile) >> eshift;
  const int npages = ((min(nmax, t_end * kTile) - 1) >> eshift) - page0 + 1;  // <= kMaxPages (host)

  uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + L::kHist);
  float* qw_s = reinterpret_cast<float*>(smem + L::kQw);
  float* qs_s = reinterpret_cast<float*>(smem + L::kQs);
  float* hw_s = reinterpret_cast<float*>(smem + L::kHw);
  int* pages_s = reinterpret_cast<int*>(smem + L::kPages);
  const uint32_t bar_full = sbase + L::kBar;
  const uint32_t bar_empty = bar_full + kStages * 8;
  const uint32_t bar_accf = bar_empty + kStages * 8;
  const uint32_t bar_acce = bar_accf + kAcc * 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  if (tid == kEpiThreads) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 33);   // the expect-tx arrival + one per producer lane
      mbar_init(bar_empty + 8 * i, 1);   // the MMA commit
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(bar_accf + 8 * i, 1);
      mbar_init(bar_acce + 8 * i, kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_k);
  }
  __syncthreads();

  if (warp == kEpiWarps) {
    tmem_alloc(sbase + L::kMisc, L::kCols);
    for (int i = lane; i < npages; i += 32) {
      const int blk = page0 + i;
      int phys = blk < p.paging.max_blocks ? p.paging.table[(long long)b * p.paging.max_blocks + blk] : -1;
      if (phys < 0 || (long long)(phys + 1) * epb > p.k_rows) {
        report(p.status, LCS_ERR_DEVICE_GUARD);
        phys = -1;
      }
      pages_s[i] = phys;
    }
  } else if (warp < kEpiWarps) {
    // ---- B operand: row n = qi*V + h*4 + blk; codes of block blk sit in 16-byte chunks 2blk, 2blk+1
    for (int idx = tid; idx < N * 8; idx += kEpiThreads) {
      const int n = idx >> 3, ch = idx & 7;
      const int qi = n / V, h = (n % V) >> 2, blk = n & 3;
      uint2 v = make_uint2(0u, 0u);
      if ((ch >> 1) == blk && qi < qn) {
        const long long qrow = (q0 + qi) * HI + h;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q_fp4 + qrow * 64 + ch * 8);
        v = make_uint2(src[0], src[1]);
      }
      const int phys_ch = ch ^ (n & 7);
      *reinterpret_cast<uint4*>(smem + L::kB + n * kRowBytes + phys_ch * 16) = make_uint4(v.x, v.y, 0u, 0u);
    }
    for (int idx = tid; idx < QPS * HI * 4; idx += kEpiThreads) {
      const int qi = idx / (HI * 4), h = (idx / 4) % HI, blk = idx % 4;
      const long long qrow = (q0 + qi) * HI + h;
      const float qsc = qi < qn ? ue8m0_to_f32(p.q_scale[qrow * 4 + blk]) : 0.0f;
      const float w = qi < qn ? (p.head_w ? p.head_w[qrow] : 1.0f) : 0.0f;
      qs_s[idx] = qsc;
      qw_s[idx] = qsc * w;   // a power of two times the head weight: exact
      if (blk == 0) hw_s[qi * HI + h] = w;
    }
    if (with_hist)
      for (int i = tid; i < QPS * kTopkHistBins / 4; i += kEpiThreads)
        reinterpret_cast<uint4*>(hist_s)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kEpiWarps && warp < kEpiWarps + kProdWarps) {
    // ---- producers (tile i by warp i % 2): lane p copies page p of the tile through the tensor
    //      map; every lane copies 16 bytes of block scales with cp.async
    for (int i = warp - kEpiWarps; i < nt; i += kProdWarps) {
      const int s = i % kStages;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar_empty + 8 * s, ((i / kStages) & 1) ^ 1, p.status, abort_flag);
      if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
      const int e0 = (t_begin + i) * kTile;
      const int rows = min(kTile, ((min(nmax, e0 + kTile) - e0 + epb - 1) >> eshift) << eshift);  // whole pages
      const uint32_t bar = bar_full + 8 * s;
      const uint32_t a_dst = sbase + L::kA + s * kATileBytes;
      const uint32_t s_dst = sbase + L::kScale + (i % kScaleSlots) * kTile * 4;
      const int npg = rows >> eshift;
      const int phys = lane < npg ? pages_s[((e0 >> eshift) - page0) + lane] : -1;
      const uint32_t valid = __ballot_sync(0xffffffffu, phys >= 0);
      if (lane == 0) mbar_arrive_expect_tx(bar, __popc(valid) * epb * kPackedRowBytes);
      __syncwarp();
      if (phys >= 0) tma_load_2d(a_dst + (lane << eshift) * kRowBytes, &tmap_k, 0, phys * epb, bar);
      const int r = lane * 4;
      const int ph = __shfl_sync(0xffffffffu, phys, (r >> eshift) & 31);
      if (r < rows && ph >= 0) cp_async16_s(s_dst + r * 4, p.k_scale + ((long long)ph * epb + (r & (epb - 1))) * 4);
      cp_async_arrive_noinc(bar);
    }
    cp_async_wait<0>();
  } else if (warp == kEpiWarps + kProdWarps) {
    if (lane == 0) {
      const uint64_t bdesc = smem_desc_sw128(sbase + L::kB);
      for (int i = 0; i < nt; ++i) {
        const int s = i % kStages, a = i % kAcc;
        if (!mbar_wait(bar_full + 8 * s, (i / kStages) & 1, p.status, abort_flag)) break;
        if (!mbar_wait(bar_acce + 8 * a, ((i / kAcc) & 1) ^ 1, p.status, abort_flag)) break;
        tc_fence_after_sync();
        const uint64_t adesc = smem_desc_sw128(sbase + L::kA + s * kATileBytes);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
          tc_mma_f8f6f4(tmem + a * N, adesc + 2 * kb, bdesc + 2 * kb, kIdesc, kb > 0 ? 1u : 0u);
        tc_commit(bar_accf + 8 * a);
        tc_commit(bar_empty + 8 * s);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32*(w%4).. (its entries) and the columns of
    //      queries QPW*(w/4) .. QPW*(w/4)+QPW-1 of every tile
    constexpr int QPW = QPS / 4;                    // queries per warp
    constexpr int CW = QPW * V;                     // their columns
    constexpr int kPhases = CW > 32 ? 2 : 1;        // column loads of at most 32 registers
    constexpr int CWP = CW / kPhases;
    static_assert(CWP % 16 == 0 && CWP <= 32 && QPW % kPhases == 0, "columns per warp");
    const int quad = warp & 3, qb = (warp >> 2) * QPW;
    const int row = quad * 32 + lane;
    const int nq_first = (n0 + qb + 1) >> mshift;   // visible entries of the warp's first query
    uint32_t* keys_row = p.keys_out != nullptr ? p.keys_out + (q0 + qb) * p.ld : nullptr;
    float* scores_row = p.scores_out != nullptr ? p.scores_out + (q0 + qb) * p.ld : nullptr;
    for (int i = 0; i < nt; ++i) {
      const int a = i % kAcc;
      bool ok = mbar_wait(bar_accf + 8 * a, (i / kAcc) & 1, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t sc = *reinterpret_cast<const uint32_t*>(smem + L::kScale + ((i % kScaleSlots) * kTile + row) * 4);
      float ksc[4];
      ksc[0] = __uint_as_float(max((sc << 23) & 0x7F800000u, 0x00400000u));
      ksc[1] = __uint_as_float(max((sc << 15) & 0x7F800000u, 0x00400000u));
      ksc[2] = __uint_as_float(max((sc << 7) & 0x7F800000u, 0x00400000u));
      ksc[3] = __uint_as_float(max((sc >> 1) & 0x7F800000u, 0x00400000u));
      const unsigned long long k01 = f2_pack(ksc[0], ksc[1]), k23 = f2_pack(ksc[2], ksc[3]);
      const int e0 = (t_begin + i) * kTile;
      const int j = e0 + row;
      const bool full = e0 + kTile <= nq_first;     // every query of the warp sees the whole tile
#pragma unroll
      for (int ph = 0; ph < kPhases; ++ph) {
        // this phase's columns into registers; the accumulator goes back after the last phase's load
        uint32_t d[CWP];
#pragma unroll
        for (int c16 = 0; c16 < CWP / 16; ++c16)
          tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + a * N + qb * V + ph * CWP + c16 * 16,
                    *reinterpret_cast<uint32_t(*)[16]>(&d[c16 * 16]));
        tmem_ld_wait();
        if (ph == kPhases - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acce + 8 * a);
        }
#pragma unroll
        for (int qp = 0; qp < QPW / kPhases; ++qp) {
          const int qq = ph * (QPW / kPhases) + qp;
          const int qi = qb + qq;
          float score;
          if (!p.relu) {
            // phi = identity: per block, the heads' weighted sum, then the block scales (every
            // term exact); blocks (0, 1) and (2, 3) in packed pairs
            unsigned long long t01 = 0ull, t23 = 0ull;
#pragma unroll
            for (int h = 0; h < HI; ++h) {
              const float4 w = *reinterpret_cast<const float4*>(qw_s + (qi * HI + h) * 4);
              const uint32_t* dh = d + qp * V + h * 4;
              t01 = f2_fma(f2_pack(__uint_as_float(dh[0]), __uint_as_float(dh[1])), f2_pack(w.x, w.y), t01);
              t23 = f2_fma(f2_pack(__uint_as_float(dh[2]), __uint_as_float(dh[3])), f2_pack(w.z, w.w), t23);
            }
            score = f2_sum(f2_fma(t23, k23, f2_mul(t01, k01)));
          } else {
            float sh[HI];
#pragma unroll
            for (int h = 0; h < HI; ++h) {
              const float4 qs = *reinterpret_cast<const float4*>(qs_s + (qi * HI + h) * 4);
              const uint32_t* dh = d + qp * V + h * 4;
              float acc = __uint_as_float(dh[0]) * (ksc[0] * qs.x);
              acc = fmaf(__uint_as_float(dh[1]), ksc[1] * qs.y, acc);
              acc = fmaf(__uint_as_float(dh[2]), ksc[2] * qs.z, acc);
              acc = fmaf(__uint_as_float(dh[3]), ksc[3] * qs.w, acc);
              sh[h] = fmaxf(acc, 0.0f) * hw_s[qi * HI + h];
            }
#pragma unroll
            for (int w = 1; w < HI; w <<= 1)
#pragma unroll
              for (int h = 0; h < HI; h += 2 * w) sh[h] = sh[h] + sh[h + w];
            score = sh[0];
          }
          if (qi < qn && (full || j < ((n0 + qi + 1) >> mshift))) {
            if (scores_row != nullptr) {
              scores_row[(long long)qq * p.ld + j] = score;
            } else {
              const uint32_t key = score_key(score);
              keys_row[(long long)qq * p.ld + j] = key;
              if (with_hist) atomicAdd(&hist_s[qi * kTopkHistBins + (key >> 21)], 1u);
            }
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kEpiWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kCols);
  } else if (warp < kEpiWarps && with_hist) {
    for (int i = tid; i < qn * kTopkHistBins; i += kEpiThreads) {
      const uint32_t c = hist_s[i];
      if (c) atomicAdd(&p.hist[(q0 + i / kTopkHistBins) * kTopkHistBins + i % kTopkHistBins], c);
    }
  }
}

namespace {

template <int HI, int QPS>
cudaError_t launch_pf_t(const CUtensorMap& tmap, const IndexParams& p, int max_new, int max_entries,
                        cudaStream_t st) {
  using L = PfSmem<HI, QPS>;
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    cudaError_t e = cudaFuncSetAttribute(index_tc_pf_kernel<HI, QPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(index_tc_pf_kernel<HI, QPS>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int tiles = (max_entries + kTile - 1) / kTile;
  if (tiles == 0) return cudaSuccess;
  const int tpc_cap = kMaxPages * p.paging.epb / kTile;   // a run spans at most kMaxPages pages
  const int runs = (tiles + tpc_cap - 1) / tpc_cap;
  const int tpc = (tiles + runs - 1) / runs;
  const int groups = (max_new + QPS - 1) / QPS;
  dim3 grid(runs, groups, p.num_seqs);
  index_tc_pf_kernel<HI, QPS><<<grid, kThreads, L::kBytes, st>>>(tmap, p, tpc);
  return cudaGetLastError();
}

}  // namespace

bool index_tc_pf_applies(const IndexParams& p, int rank, int max_new) {
  if (rank != 128 || p.paging.epb < 8 || p.paging.epb > 128 || (p.paging.epb & (p.paging.epb - 1))) return false;
  if ((reinterpret_cast<uintptr_t>(p.k_fp4) & 31u) || (reinterpret_cast<uintptr_t>(p.k_scale) & 15u)) return false;
  if (p.k_rows < p.paging.epb || p.k_rows > (1ll << 31)) return false;
  if (max_new <= 4 || (max_new + 7) / 8 > 65535) return false;
  return p.heads == 1 || p.heads == 2 || p.heads == 4 || p.heads == 8;
}

cudaError_t launch_index_tc_pf(const IndexParams& p, int rank, int max_new, int max_entries, cudaStream_t st) {
  if (!index_tc_pf_applies(p, rank, max_new)) return cudaErrorInvalidValue;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)rank, (cuuint64_t)p.k_rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)(rank / 2)};
  const cuuint32_t box[2] = {128u, (cuuint32_t)p.paging.epb};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(p.k_fp4), gdim, gstride, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  switch (p.heads) {
    case 1: return launch_pf_t<1, 16>(tmap, p, max_new, max_entries, st);
    case 2: return launch_pf_t<2, 16>(tmap, p, max_new, max_entries, st);
    case 4: return launch_pf_t<4, 16>(tmap, p, max_new, max_entries, st);
    case 8: return launch_pf_t<8, 8>(tmap, p, max_new, max_entries, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lcsa
