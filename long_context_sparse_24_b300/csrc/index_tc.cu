// Lightning-indexer scores on the tcgen05 tensor cores for batches with a few
// queries per sequence (decode, short speculative runs).
//
// Defined by: m.x-techcon.com/article/133366, section 2, CSA step 2 (a low-rank indexer scores
// every compressed entry, each query keeps its top-k) and section 4 "FP4量化感知训练" (the
// indexer's QK path runs in FP4).  Same arithmetic as the warp-MMA scorer in indexer.cu:
//   score(q, j) = sum_h w[q,h] * phi( sum_blk 2^(eq[q,h,blk] + ek[j,blk]) * dot_blk(q_h, k_j) ).
//
// Layout of the work.  A persistent, warp-specialised CTA scans a contiguous run of 128-entry
// tiles of one sequence for all of that sequence's queries (QPS <= 4), through a ring of
// shared-memory stages:
//   warps 8-9 (producers, alternating tiles) look the run's pages up in the block table once, then streams tiles:
//                      one lane per page issues a TMA copy of the page's codes in the tensor
//                      map's "16 x U4 in 16 bytes" form with the 128-byte swizzle -- each
//                      entry's 128 E2M1 codes occupy one 128-byte shared-memory row, the K-major
//                      operand form of the kind::f8f6f4 MMA with E2M1 inputs -- and every lane
//                      copies 16 bytes of block scales with cp.async (tiny bulk copies issue too
//                      slowly from one thread to keep a paged scan at memory speed);
//   warp 10 (MMA)       issues four K = 32 MMAs per tile into one of kAcc tensor-memory
//                      accumulators and commits them to that accumulator's barrier;
//   warps 0-7          (one thread per entry = per TMEM lane, two warps per lane quadrant
//                      taking alternate tiles) read the accumulator and release it, form the scores, write the order-preserving keys and
//                      count them into the per-query key histogram used by the top-k selection.
// The grid is one wave: about (SMs x resident CTAs) / sequences CTAs per sequence.
//
// The MMA: A = 128 entries x 128 codes, B = N rows built from the queries, where row
// (blk, q, h) holds query q's head-h codes inside block blk and zeros elsewhere.  Four MMAs of
// K = 32 (one per block) accumulate into D = 128 x N fp32 in tensor memory; because every B row
// is zero outside its block, column (blk, q, h) of D is exactly that block's partial dot product
// (a sum of 32 products of E2M1 values: multiples of 1/4 below 2^11, exact in fp32).  Block
// scales and head weights are applied afterwards in fp32, as in the warp-MMA scorer.
#include "kernels.cuh"
#include "sm100.cuh"

namespace lcsa {

namespace {

constexpr int kTile = 128;          // entries per MMA tile (M)
#ifndef LCSA_INDEX_STAGES
#define LCSA_INDEX_STAGES 5
#endif
constexpr int kStages = LCSA_INDEX_STAGES;  // shared-memory ring depth (tiles in flight per CTA)
constexpr int kAcc = 4;             // tensor-memory accumulators
constexpr int kMaxPages = 256;      // block-table entries a CTA's run may span
constexpr int kRowBytes = 128;      // shared-memory bytes of one entry's 128 codes (16U4 in 16 B)
constexpr int kPackedRowBytes = 64; // global bytes of the same codes
constexpr int kATileBytes = kTile * kRowBytes;
constexpr int kEpiWarps = 8;        // two per TMEM lane quadrant, alternating tiles
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kProdWarps = 2;       // producer warps, alternating tiles
constexpr int kScaleSlots = 2 * kStages;  // block-scale ring (read by the epilogue, outlives a stage)
constexpr int kThreads = kEpiThreads + 32 * kProdWarps + 32;

template <int QH, int QPS>
struct TcSmem {
  static constexpr int N = 4 * QH;                            // MMA N: (block, query-head) columns
  static constexpr int kA = 0;                                // kStages x 16 KB, 1024-aligned
  static constexpr int kB = kA + kStages * kATileBytes;       // N x 128 B
  static constexpr int kScale = kB + N * kRowBytes;           // kScaleSlots x 128 x 4 B
  static constexpr int kQs = kScale + kScaleSlots * kTile * 4;  // f32 [QH][4] q block scales
  static constexpr int kHw = kQs + QH * 4 * 4;                // f32 [QH] head weights
  static constexpr int kPages = kHw + QH * 4;                 // int [kMaxPages]
  static constexpr int kBar = kPages + kMaxPages * 4;         // u64 full/empty[kStages], accf/acce[kAcc]
  static constexpr int kMisc = kBar + (2 * kStages + 2 * kAcc) * 8;  // tmem base, abort flag
  static constexpr int kHist = kMisc + 16;                    // u32 [QPS][2048]
  static constexpr int kBytes = kHist + QPS * kTopkHistBins * 4 + 1024;
};

__host__ __device__ constexpr uint32_t tmem_cols_for(int n) {
  const int c = kAcc * n;
  return c <= 32 ? 32 : (c <= 64 ? 64 : (c <= 128 ? 128 : (c <= 256 ? 256 : 512)));
}

}  // namespace

// grid: (runs per sequence, num_seqs); block kThreads.  CTA (x, b) scans tiles
// [x*tiles_per_cta, (x+1)*tiles_per_cta) of sequence b (clipped to its visible entries).
template <int HI, int QH>
__global__ void __launch_bounds__(kThreads) index_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, IndexParams p,
                                                           int tiles_per_cta) {
  constexpr int QPS = QH / HI;
  using L = TcSmem<QH, QPS>;
  constexpr int N = L::N;
  constexpr uint32_t kCols = tmem_cols_for(N);
  constexpr uint32_t kIdesc = idesc_f8f6f4(5, 5, kTile, N);  // E2M1 x E2M1 -> f32, M = 128
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int qn = min(sp.qn, QPS);
  if (qn <= 0) return;
  const int n0 = sp.n0();
  const int mshift = 31 - __clz(p.m);
  const int nmax = (n0 + qn) >> mshift;          // visible entries of the sequence's last query
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
      mbar_init(bar_acce + 8 * i, 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_k);
  }
  __syncthreads();

  if (warp == kEpiWarps) {
    tmem_alloc(sbase + L::kMisc, kCols);
    // physical block of every page the run touches (-1: unmapped or outside the key rows)
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
    // ---- B operand: row n = blk*QH + c, c = qi*HI + h; codes of block blk in chunks 2blk, 2blk+1
    for (int idx = tid; idx < N * 8; idx += kEpiThreads) {
      const int n = idx >> 3, ch = idx & 7;
      const int blk = n / QH, c = n % QH;
      const int qi = c / HI, h = c % HI;
      uint2 v = make_uint2(0u, 0u);
      if ((ch >> 1) == blk && qi < qn) {
        const long long qrow = (long long)(sp.q0 + qi) * HI + h;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q_fp4 + qrow * 64 + ch * 8);
        v = make_uint2(src[0], src[1]);
      }
      const int phys_ch = ch ^ (n & 7);
      *reinterpret_cast<uint4*>(smem + L::kB + n * kRowBytes + phys_ch * 16) = make_uint4(v.x, v.y, 0u, 0u);
    }
    for (int idx = tid; idx < QH * 4; idx += kEpiThreads) {
      const int c = idx >> 2, blk = idx & 3;
      const int qi = c / HI, h = c % HI;
      qs_s[idx] = qi < qn ? ue8m0_to_f32(p.q_scale[((long long)(sp.q0 + qi) * HI + h) * 4 + blk]) : 0.0f;
    }
    for (int c = tid; c < QH; c += kEpiThreads) {
      const int qi = c / HI, h = c % HI;
      hw_s[c] = qi < qn ? (p.head_w ? p.head_w[(long long)(sp.q0 + qi) * HI + h] : 1.0f) : 0.0f;
    }
    if (with_hist)
      for (int i = tid; i < qn * kTopkHistBins; i += kEpiThreads) hist_s[i] = 0u;
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kEpiWarps && warp < kEpiWarps + kProdWarps) {
    // ---- producer warps (tile i by producer warp i % kProdWarps): stage i % kStages receives
    //      tile t_begin + i.  Lane p issues page p's
    //      tensor copy of the codes (the TMA unpacks them into the MMA operand form); every lane
    //      copies 16 bytes of block scales with cp.async.  The stage's barrier expects the code
    //      bytes from the copies plus one arrival per lane when its scale copy lands.
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
      const int r = lane * 4;   // this lane's four scale words
      const int ph = __shfl_sync(0xffffffffu, phys, (r >> eshift) & 31);
      if (r < rows && ph >= 0) cp_async16_s(s_dst + r * 4, p.k_scale + ((long long)ph * epb + (r & (epb - 1))) * 4);
      cp_async_arrive_noinc(bar);
    }
    cp_async_wait<0>();
  } else if (warp == kEpiWarps + kProdWarps) {
    if (lane == 0) {
      // ---- MMA issuer: tile i -> accumulator i % kAcc
      const uint64_t bdesc = smem_desc_sw128(sbase + L::kB);
      for (int i = 0; i < nt; ++i) {
        const int s = i % kStages, a = i % kAcc;
        if (!mbar_wait(bar_full + 8 * s, (i / kStages) & 1, p.status, abort_flag)) break;
        if (!mbar_wait(bar_acce + 8 * a, ((i / kAcc) & 1) ^ 1, p.status, abort_flag)) break;
        tc_fence_after_sync();
        const uint64_t adesc = smem_desc_sw128(sbase + L::kA + s * kATileBytes);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)   // K = 32 codes per MMA: 32 shared-memory bytes per step
          tc_mma_f8f6f4(tmem + a * N, adesc + 2 * kb, bdesc + 2 * kb, kIdesc, kb > 0 ? 1u : 0u);
        tc_commit(bar_accf + 8 * a);
        tc_commit(bar_empty + 8 * s);   // the stage is free once these MMAs have read it
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32*(w%4).. of the tiles i with i % 2 == w / 4
    const int quad = warp & 3, par = warp >> 2;
    float qsc[QH][4], hw[QH], qw[QH][4];
#pragma unroll
    for (int c = 0; c < QH; ++c) {
      hw[c] = hw_s[c];
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        qsc[c][blk] = qs_s[c * 4 + blk];
        qw[c][blk] = qsc[c][blk] * hw[c];   // powers of two times the head weight: exact
      }
    }
    int nq[QPS];
#pragma unroll
    for (int qi = 0; qi < QPS; ++qi) nq[qi] = qi < qn ? (n0 + qi + 1) >> mshift : 0;
    const int row = quad * 32 + lane;
    for (int i = par; i < nt; i += 2) {
      const int a = i % kAcc;
      bool ok = mbar_wait(bar_accf + 8 * a, (i / kAcc) & 1, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t d[N];
#pragma unroll
      for (int c16 = 0; c16 < N / 16; ++c16)
        tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + a * N + c16 * 16,
                  *reinterpret_cast<uint32_t(*)[16]>(&d[c16 * 16]));
      tmem_ld_wait();
      const uint32_t sc = *reinterpret_cast<const uint32_t*>(smem + L::kScale + ((i % kScaleSlots) * kTile + row) * 4);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce + 8 * a);
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
            for (int h = 0; h < HI; ++h) t = fmaf(__uint_as_float(d[blk * QH + qi * HI + h]), qw[qi * HI + h][blk], t);
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
            for (int blk = 0; blk < 4; ++blk) acc = fmaf(__uint_as_float(d[blk * QH + c]), ksc[blk] * qsc[c][blk], acc);
            sh[h] = fmaxf(acc, 0.0f) * hw[c];
          }
#pragma unroll
          for (int w = 1; w < HI; w <<= 1)
#pragma unroll
            for (int h = 0; h < HI; h += 2 * w) sh[h] = sh[h] + sh[h + w];
          score = sh[0];
        }
        if (j < nq[qi]) {
          const long long o = (long long)(sp.q0 + qi) * p.ld + j;
          if (p.scores_out != nullptr) {
            p.scores_out[o] = score;
          } else {
            const uint32_t key = score_key(score);
            p.keys_out[o] = key;
            if (with_hist) atomicAdd(&hist_s[qi * kTopkHistBins + (key >> 21)], 1u);
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kEpiWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kCols);
  } else if (warp < kEpiWarps && with_hist) {
    for (int i = tid; i < qn * kTopkHistBins; i += kEpiThreads) {
      const uint32_t c = hist_s[i];
      if (c) atomicAdd(&p.hist[(long long)(sp.q0 + i / kTopkHistBins) * kTopkHistBins + i % kTopkHistBins], c);
    }
  }
}

// ----------------------------------------------------------------------------------------------
// launcher
// ----------------------------------------------------------------------------------------------

namespace {

template <int HI, int QH>
cudaError_t launch_tc_t(const CUtensorMap& tmap, const IndexParams& p, int max_entries, int sms, cudaStream_t st) {
  using L = TcSmem<QH, QH / HI>;
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<HI, QH>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(index_tc_kernel<HI, QH>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  // resident CTAs per SM: shared memory (228 KB per SM, 1 KB reserved per CTA) and tensor memory
  int occ = (228 * 1024) / (L::kBytes + 1024);
  const int occ_tmem = 512 / (int)tmem_cols_for(L::N);
  if (occ > occ_tmem) occ = occ_tmem;
  if (occ < 1) occ = 1;
  const int tiles = (max_entries + kTile - 1) / kTile;
  if (tiles == 0) return cudaSuccess;
  int runs = (sms * occ) / p.num_seqs;             // one wave of CTAs
  if (runs < 1) runs = 1;
  int tpc = (tiles + runs - 1) / runs;
  const int tpc_cap = kMaxPages * p.paging.epb / kTile;   // a run spans at most kMaxPages pages
  if (tpc > tpc_cap) tpc = tpc_cap;
  dim3 grid((tiles + tpc - 1) / tpc, p.num_seqs);
  index_tc_kernel<HI, QH><<<grid, kThreads, L::kBytes, st>>>(tmap, p, tpc);
  return cudaGetLastError();
}

}  // namespace

// Columns (query-heads) per 32-code block the tensor-core scorer needs, or 0 when it does not
// apply (rank other than 128, pages outside 8..128 entries, more than 4 queries per sequence,
// key codes not 32-byte or scales not 16-byte aligned).
int index_tc_qh(const IndexParams& p, int rank, int max_new) {
  if (rank != 128 || p.paging.epb < 8 || p.paging.epb > 128 || (p.paging.epb & (p.paging.epb - 1))) return 0;
  if ((reinterpret_cast<uintptr_t>(p.k_fp4) & 31u) || (reinterpret_cast<uintptr_t>(p.k_scale) & 15u)) return 0;
  if (p.k_rows < p.paging.epb || p.k_rows > (1ll << 31)) return 0;
  if (max_new < 1 || max_new > 4) return 0;
  const int need = max_new * p.heads;
  const int qh = need <= 4 ? 4 : (need <= 8 ? 8 : (need <= 16 ? 16 : 0));
  if (qh == 0 || qh / p.heads < max_new) return 0;
  return qh;
}

cudaError_t launch_index_tc(const IndexParams& p, int rank, int max_new, int max_entries, int sms, cudaStream_t st) {
  const int qh = index_tc_qh(p, rank, max_new);
  if (qh == 0) return cudaErrorInvalidValue;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // codes as [rows][128] 4-bit values; a box of one page is unpacked to 16 codes per 16 bytes
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)rank, (cuuint64_t)p.k_rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)(rank / 2)};
  const cuuint32_t box[2] = {128u, (cuuint32_t)p.paging.epb};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(p.k_fp4), gdim, gstride, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  switch (p.heads * 100 + qh) {
    case 104: return launch_tc_t<1, 4>(tmap, p, max_entries, sms, st);
    case 204: return launch_tc_t<2, 4>(tmap, p, max_entries, sms, st);
    case 208: return launch_tc_t<2, 8>(tmap, p, max_entries, sms, st);
    case 404: return launch_tc_t<4, 4>(tmap, p, max_entries, sms, st);
    case 408: return launch_tc_t<4, 8>(tmap, p, max_entries, sms, st);
    case 416: return launch_tc_t<4, 16>(tmap, p, max_entries, sms, st);
    case 808: return launch_tc_t<8, 8>(tmap, p, max_entries, sms, st);
    case 816: return launch_tc_t<8, 16>(tmap, p, max_entries, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lcsa
