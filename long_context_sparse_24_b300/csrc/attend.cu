// Shared-KV multi-query attention over gathered rows (CSA: top-k entries + window; HCA: every
// visible entry + window).
//
// Defined by: m.x-techcon.com/article/133366, section 2: CSA step 3 (the selected compressed
// entries and the most recent 128 uncompressed tokens are attended together) and the HCA
// paragraph (dense attention over every entry, the same window, shared-KV multi-query
// attention); the efficiency paragraph fixes the row storage (RoPE dims BF16, the rest FP8).
//
// One CTA handles one query token, one group of 16*MT heads and one split of its row list.
// Per tile of RT=32 rows:
//   gather   cp.async copies of the rows' stored bytes (FP8 codes, BF16 RoPE dims, fp32 scale)
//            into a staging buffer, two stages deep;
//   widen    FP8 codes -> f16 (exact), RoPE dims kept BF16, into a swizzled [RT][D] tile;
//   S = QK^T two accumulators per logit: BF16 MMA over the 64 RoPE dims, f16 MMA over the FP8
//            dims (query converted to f16 once); logit = s_rope + scale_row * s_fp8, so the FP8
//            row scale is applied exactly once in fp32;
//   softmax  online, in base 2, fp32; P (bf16) for the RoPE output dims and P*scale_row*2^8
//            (f16) for the FP8 output dims;
//   O += PV  every warp owns D/8 output columns for all heads of the CTA.
// Separate values (SV): the stage holds the value rows' bytes next to the key rows'; once S is
// computed the value rows are widened into the same tile and P2 takes the value row's scale.
// Splits write (O, m, l) partials that a second kernel combines with the usual LSE rule.
#include "kernels.cuh"

namespace lcsa {

constexpr int kRT = 32;           // rows per tile
constexpr int kStages = 3;        // cp.async gather stages in flight
constexpr int kDescRows = 256;    // row descriptors resolved per refill (8 tiles)
constexpr float kP2Scale = 256.f; // power-of-two pre-scale of P*scale_row for the f16 operand



__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async4_zfill(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] 16-bit tile (D/8 >= 8 chunks per row).
template <int D>
__device__ __forceinline__ int tile_off(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}
// Same for the [HG][RT] probability tiles (4 chunks per row).
__device__ __forceinline__ int ptile_off(int r, int c) { return r * (kRT * 2) + ((c ^ ((r >> 1) & 3)) << 4); }

// One stage: the key rows' stored bytes (codes / RoPE dims / scales), with SV the value rows' in
// the same layout at kV, then the row-valid flags.
template <int D, int FMT, bool SV>
struct StageLayout {
  static constexpr int kNopeBytes = FMT == LCS_ROW_FP8_SPLIT ? (D - kRope) : D * 2;
  static constexpr int kRopeBytes = FMT == LCS_ROW_FP8_SPLIT ? kRope * 2 : 0;
  static constexpr int kNope = 0;
  static constexpr int kRopeOff = kRT * kNopeBytes;
  static constexpr int kScaleOff = kRopeOff + kRT * kRopeBytes;
  static constexpr int kPart = (kScaleOff + kRT * 4 + 127) / 128 * 128;
  static constexpr int kV = kPart;
  static constexpr int kValidOff = kPart * (SV ? 2 : 1);
  static constexpr int kBytes = ((kValidOff + kRT * 4) + 127) / 128 * 128;
};

template <int D, int FMT, int MT, bool SV = false>
struct AttendSmem {
  static constexpr int HG = 16 * MT;
  static constexpr int kQ = 0;
  static constexpr int kR = kQ + HG * D * 2;
  static constexpr int kStage = kR + kRT * D * 2;
  static constexpr int kS = kStage + kStages * StageLayout<D, FMT, SV>::kBytes;
  static constexpr int kSStride = kRT + 1;
  static constexpr int kP = kS + HG * kSStride * 4;
  static constexpr int kP2 = kP + HG * kRT * 2;
  static constexpr int kRowScale = kP2 + HG * kRT * 2;
  static constexpr int kVScale = kRowScale + kRT * 4;      // SV: the value rows' scales
  static constexpr int kM = kVScale + (SV ? kRT * 4 : 0);
  static constexpr int kL = kM + HG * 4;
  static constexpr int kAlpha = kL + HG * 4;
  static constexpr int kDesc = kAlpha + HG * 4;              // long long [kDescRows]
  static constexpr int kBytes = kDesc + kDescRows * 8;
};

// Locate sequence of global query q (cu_new non-decreasing).
__device__ __forceinline__ int find_seq(const int32_t* cu_new, int num_seqs, int q) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu_new[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int D, int FMT, int MT, bool SV>
__global__ void __launch_bounds__(256, 1) attend_kernel(AttendParams p) {
  using L = AttendSmem<D, FMT, MT, SV>;
  using SL = StageLayout<D, FMT, SV>;
  constexpr int HG = L::HG;
  constexpr bool kSplitFmt = FMT == LCS_ROW_FP8_SPLIT;
  constexpr int kChunks = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int q = blockIdx.x, hg = blockIdx.y, split = blockIdx.z;
  const int H = p.heads;
  const int b = find_seq(p.cu_new, p.num_seqs, q);
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int n0 = sp.n0();
  const int t = n0 + (q - sp.q0);
  int cnt;
  const int32_t* sel = nullptr;
  if (p.topk_idx != nullptr) {
    sel = p.topk_idx + (long long)q * p.k;
    if (p.topk_cnt != nullptr) {
      cnt = min(p.topk_cnt[q], p.k);
    } else {
      cnt = 0;
      while (cnt < p.k && sel[cnt] >= 0) ++cnt;
    }
  } else {
    cnt = (t + 1) / p.m;
  }
  const int nvis = (t + 1) / p.m;
  const int W = min(t + 1, kWindow);
  const int R = cnt + W;
  const int r_begin = split * p.rows_per_split;
  const int r_end = min(R, r_begin + p.rows_per_split);
  const int h0 = hg * HG;

  float* mrow = reinterpret_cast<float*>(smem + L::kM);
  float* lrow = reinterpret_cast<float*>(smem + L::kL);
  float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);

  if (r_begin >= r_end) {
    // empty split: mark it for the combine step
    if (p.splits > 1) {
      for (int h = tid; h < HG; h += 256)
        if (h0 + h < H) {
          float* ml = p.ws_ml + (((long long)q * H + h0 + h) * p.splits + split) * 2;
          ml[0] = -INFINITY;
          ml[1] = 0.0f;
        }
    }
    return;
  }

  // ---- row descriptors: source set (bits 60..61: 0 entries, 1 new rows, 2 window ring; -1 =
  //      invalid) and physical row, resolved for kDescRows rows at a time so that the gather of a
  //      tile issues its copies without waiting on index loads
  long long* desc = reinterpret_cast<long long*>(smem + L::kDesc);
  auto fill_descs = [&](int seg_begin) {
    const int r = seg_begin + tid;
    long long d = -1;
    if (r < r_end) {
      if (r < cnt) {
        const int j = sel ? sel[r] : r;
        long long row = -1;
        if (j >= 0 && j < nvis) row = entry_row(p.paging, b, j, p.entries.num_rows);
        if (row < 0) report(p.status, LCS_ERR_DEVICE_GUARD);
        d = row;
      } else {
        const int pos = t - W + 1 + (r - cnt);
        long long row;
        if (pos >= n0 && p.new_rows.nope != nullptr) {
          row = (long long)sp.q0 + (pos - n0);
          d = row < p.new_rows.num_rows ? (row | (1ll << 60)) : -1;
        } else {
          row = (long long)b * kWindow + (pos % kWindow);
          d = row < p.window.num_rows ? (row | (2ll << 60)) : -1;
        }
        if (d < 0) report(p.status, LCS_ERR_DEVICE_GUARD);
      }
    }
    if (tid < kDescRows) desc[tid] = d;
  };

  // ---- gather issue: thread -> (row rr = tid/8, sub u = tid%8)
  auto issue_tile = [&](int tile_begin, int stage) {
    uint8_t* st = smem + L::kStage + stage * SL::kBytes;
    const int rr = tid >> 3, u = tid & 7;
    const int r = tile_begin + rr;
    const long long d = r < r_end ? desc[(r - r_begin) % kDescRows] : -1;
    const bool ok = d >= 0;
    const int kind = ok ? (int)(d >> 60) : 0;
    const long long rw = ok ? (d & ((1ll << 60) - 1)) : 0;
    const uint8_t* src_nope = kind == 1 ? p.new_rows.nope : (kind == 2 ? p.window.nope : p.entries.nope);
    const uint8_t* src_rope = reinterpret_cast<const uint8_t*>(kind == 1 ? p.new_rows.rope
                                                               : (kind == 2 ? p.window.rope : p.entries.rope));
    const float* src_scale = kind == 1 ? p.new_rows.scale : (kind == 2 ? p.window.scale : p.entries.scale);
    const int nb = ok ? 16 : 0;   // invalid rows are zero-filled from row 0 of a set that has one
    for (int c = u; c < SL::kNopeBytes / 16; c += 8)
      cp_async16_zfill(st + rr * SL::kNopeBytes + c * 16, src_nope + rw * SL::kNopeBytes + c * 16, nb);
    if (kSplitFmt) {
      cp_async16_zfill(st + SL::kRopeOff + rr * SL::kRopeBytes + u * 16, src_rope + rw * SL::kRopeBytes + u * 16, nb);
      if (u == 0) cp_async4_zfill(st + SL::kScaleOff + rr * 4, src_scale + rw, ok ? 4 : 0);
    }
    if (SV) {   // the value row with the same number in the matching value set
      const Rows& vs = kind == 1 ? p.v_new_rows : (kind == 2 ? p.v_window : p.v_entries);
      uint8_t* sv = st + SL::kV;
      for (int c = u; c < SL::kNopeBytes / 16; c += 8)
        cp_async16_zfill(sv + rr * SL::kNopeBytes + c * 16, vs.nope + rw * SL::kNopeBytes + c * 16, nb);
      if (kSplitFmt) {
        cp_async16_zfill(sv + SL::kRopeOff + rr * SL::kRopeBytes + u * 16,
                         reinterpret_cast<const uint8_t*>(vs.rope) + rw * SL::kRopeBytes + u * 16, nb);
        if (u == 0) cp_async4_zfill(sv + SL::kScaleOff + rr * 4, vs.scale + rw, ok ? 4 : 0);
      }
    }
    if (u == 0) reinterpret_cast<int*>(st + SL::kValidOff)[rr] = ok ? 1 : 0;
  };

  const int ntiles = (r_end - r_begin + kRT - 1) / kRT;
  constexpr int kTilesPerSeg = kDescRows / kRT;
  fill_descs(r_begin);
  __syncthreads();

  // ---- Q tile -> shared with cp.async (one batch of 16-byte copies); FP8-split rows: the
  //      non-RoPE dims are converted to f16 in place once the copies have landed (tile 0)
  {
    uint8_t* Qs = smem + L::kQ;
    for (int idx = tid; idx < HG * kChunks; idx += 256) {
      const int h = idx / kChunks, c = idx % kChunks;
      uint8_t* dst = Qs + tile_off<D>(h, c);
      if (h0 + h < H) cp_async16(dst, p.q + ((long long)q * H + h0 + h) * D + c * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
    for (int h = tid; h < HG; h += 256) {
      mrow[h] = -INFINITY;
      lrow[h] = 0.0f;
    }
  }

  for (int pre = 0; pre < kStages - 1; ++pre) {
    if (pre < ntiles) issue_tile(r_begin + pre * kRT, pre);
    cp_async_commit();
  }

  // ---- output accumulators: warp owns columns [warp*D/8, (warp+1)*D/8)
  constexpr int DW = D / 8;          // columns per warp
  constexpr int NTD = DW / 8;        // n8 tiles per warp
  float oacc[MT][NTD][4];
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int c = 0; c < NTD; ++c)
#pragma unroll
      for (int k = 0; k < 4; ++k) oacc[a][c][k] = 0.0f;
  const int dcol0 = warp * DW;
  const bool warp_rope = kSplitFmt && dcol0 < kRope;   // the warp's columns are all RoPE dims

  uint8_t* Rs = smem + L::kR;
  float* Sb = reinterpret_cast<float*>(smem + L::kS);
  uint8_t* Ps = smem + L::kP;
  uint8_t* P2s = smem + L::kP2;
  float* rscale = reinterpret_cast<float*>(smem + L::kRowScale);

  for (int ti = 0; ti < ntiles; ++ti) {
    const int tile_begin = r_begin + ti * kRT;
    {
      const int nx = ti + kStages - 1;            // tile to issue now
      if (nx < ntiles && nx % kTilesPerSeg == 0) {  // its rows start a new descriptor segment
        __syncthreads();                          // every earlier issue has read the old ones
        fill_descs(r_begin + nx * kRT);
        __syncthreads();
      }
      if (nx < ntiles) issue_tile(r_begin + nx * kRT, nx % kStages);
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();

    if (kSplitFmt && ti == 0) {
      uint8_t* Qs = smem + L::kQ;
      constexpr int kNopeChunks = kChunks - kRope / 8;
      for (int idx = tid; idx < HG * kNopeChunks; idx += 256) {
        const int h = idx / kNopeChunks, c = kRope / 8 + idx % kNopeChunks;
        uint32_t* w = reinterpret_cast<uint32_t*>(Qs + tile_off<D>(h, c));
        uint4 v = *reinterpret_cast<uint4*>(w);
        uint32_t* x = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x[k]));
          __half2 hh = __float22half2_rn(f);
          x[k] = *reinterpret_cast<uint32_t*>(&hh);
        }
        *reinterpret_cast<uint4*>(w) = v;
      }
    }
    // ---- widen the staged rows (key rows, then with SV the value rows) into the [RT][D] tile
    const uint8_t* st = smem + L::kStage + (ti % kStages) * SL::kBytes;
    auto widen = [&](const uint8_t* src) {
      for (int idx = tid; idx < kRT * kChunks; idx += 256) {
        const int r = idx / kChunks, c = idx % kChunks;
        uint4 v;
        if (!kSplitFmt) {
          v = *reinterpret_cast<const uint4*>(src + r * SL::kNopeBytes + c * 16);
        } else if (c < kRope / 8) {
          v = *reinterpret_cast<const uint4*>(src + SL::kRopeOff + r * SL::kRopeBytes + c * 16);
        } else {
          const uint2 raw = *reinterpret_cast<const uint2*>(src + r * SL::kNopeBytes + (c - kRope / 8) * 8);
          v.x = e4m3x2_to_f16x2(raw.x & 0xFFFF);
          v.y = e4m3x2_to_f16x2(raw.x >> 16);
          v.z = e4m3x2_to_f16x2(raw.y & 0xFFFF);
          v.w = e4m3x2_to_f16x2(raw.y >> 16);
        }
        *reinterpret_cast<uint4*>(Rs + tile_off<D>(r, c)) = v;
      }
    };
    widen(st);
    const int* valid = reinterpret_cast<const int*>(st + SL::kValidOff);
    if (tid < kRT) {
      const bool ok = valid[tid] != 0 && tile_begin + tid < r_end;
      float sc = ok ? (kSplitFmt ? reinterpret_cast<const float*>(st + SL::kScaleOff)[tid] : 1.0f) : -1.0f;
      if (ok && kSplitFmt && !(sc < kMaxRowScale)) {   // P * s * 2^8 would leave the f16 range
        report(p.status, LCS_ERR_DEVICE_GUARD);
        sc = -1.0f;
      }
      if (SV) {
        // the value row's scale weights P2; a value row outside the bound leaves the row out
        float vsc = ok ? (kSplitFmt ? reinterpret_cast<const float*>(st + SL::kV + SL::kScaleOff)[tid] : 1.0f) : -1.0f;
        if (ok && kSplitFmt && !(vsc < kMaxRowScale)) {
          report(p.status, LCS_ERR_DEVICE_GUARD);
          sc = -1.0f;
        }
        reinterpret_cast<float*>(smem + L::kVScale)[tid] = vsc;
      }
      rscale[tid] = sc;
    }
    __syncthreads();

    // ---- S = Q R^T  (MT m-tiles x RT/8 n-tiles spread over 8 warps)
    {
      constexpr int NTILES = kRT / 8;
      constexpr int PAIRS = MT * NTILES;
      constexpr int NTW = PAIRS >= 8 ? PAIRS / 8 : 1;
      constexpr int ACTIVE = PAIRS / NTW;
      if (warp < ACTIVE) {
        const int pair0 = warp * NTW;
        const int mt = pair0 / NTILES, nt0 = pair0 % NTILES;
        float sr[NTW][4], sn[NTW][4];
#pragma unroll
        for (int a = 0; a < NTW; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k) sr[a][k] = sn[a][k] = 0.0f;
        const uint32_t qbase = smem_u32(smem + L::kQ);
        const uint32_t rbase = smem_u32(Rs);
#pragma unroll 4
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          {
            const int i = lane;
            const int row = mt * 16 + (i & 7) + ((i >> 3) & 1) * 8;
            const int ch = kk * 2 + (i >> 4);
            ldsm_x4(qbase + tile_off<D>(row, ch), a0, a1, a2, a3);
          }
#pragma unroll
          for (int a = 0; a < NTW; ++a) {
            uint32_t b0, b1;
            const int i = lane & 15;
            const int row = (nt0 + a) * 8 + (i & 7);
            const int ch = kk * 2 + (i >> 3);
            ldsm_x2(rbase + tile_off<D>(row, ch), b0, b1);
            if (kSplitFmt && kk >= kRope / 16) mma_f16(sn[a], a0, a1, a2, a3, b0, b1);
            else mma_bf16(sr[a], a0, a1, a2, a3, b0, b1);
          }
        }
#pragma unroll
        for (int a = 0; a < NTW; ++a) {
          const int col = (nt0 + a) * 8 + 2 * t4;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = col + (k & 1);
            const int hrow = mt * 16 + g + (k >> 1) * 8;
            const float s = rscale[c];
            float v = kSplitFmt ? fmaf(s, sn[a][k], sr[a][k]) : sr[a][k];
            v = s < 0.0f ? -INFINITY : v * p.scale_log2;
            Sb[hrow * L::kSStride + c] = v;
          }
        }
      }
    }
    __syncthreads();

    // the S MMAs have read the key rows: the value rows take their place (the softmax below
    // touches neither)
    if (SV) widen(st + SL::kV);

    // ---- online softmax over this tile
    {
      constexpr int TPH = 256 / HG;      // threads per head row
      constexpr int CPT = kRT / TPH;     // columns per thread
      const int h = tid / TPH, c0 = (tid % TPH) * CPT;
      float sv[CPT];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        sv[c] = Sb[h * L::kSStride + c0 + c];
        mx = fmaxf(mx, sv[c]);
      }
#pragma unroll
      for (int o = 1; o < TPH; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = mrow[h];
      const float m_new = fmaxf(m_old, mx);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.0f : exp2f(m_old - m_new);
      float sum = 0.0f;
      uint16_t pb[CPT], p2[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const float pv = none ? 0.0f : exp2f(sv[c] - m_new);
        sum += pv;
        const __nv_bfloat16 bb = __float2bfloat16_rn(pv);
        pb[c] = *reinterpret_cast<const uint16_t*>(&bb);
        const float s = SV ? reinterpret_cast<const float*>(smem + L::kVScale)[c0 + c] : rscale[c0 + c];
        const __half hh = __float2half_rn(fminf(pv * fmaxf(s, 0.0f) * kP2Scale, 65504.0f));
        p2[c] = *reinterpret_cast<const uint16_t*>(&hh);
      }
#pragma unroll
      for (int o = 1; o < TPH; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      // write P / P2 (CPT consecutive 16-bit values; CPT is 8 or 2)
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int col = c0 + c;
        const int off = ptile_off(h, col >> 3) + (col & 7) * 2;
        *reinterpret_cast<uint16_t*>(Ps + off) = pb[c];
        *reinterpret_cast<uint16_t*>(P2s + off) = p2[c];
      }
      __syncwarp();
      if ((tid % TPH) == 0) {
        mrow[h] = m_new;
        lrow[h] = lrow[h] * alpha + sum;
        alpha_s[h] = alpha;
      }
    }
    __syncthreads();

    // ---- O = alpha * O + P V
    {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const float al0 = alpha_s[mt * 16 + g], al1 = alpha_s[mt * 16 + g + 8];
#pragma unroll
        for (int c = 0; c < NTD; ++c) {
          oacc[mt][c][0] *= al0;
          oacc[mt][c][1] *= al0;
          oacc[mt][c][2] *= al1;
          oacc[mt][c][3] *= al1;
        }
      }
      const uint32_t pbase = smem_u32(kSplitFmt && !warp_rope ? P2s : Ps);
      const uint32_t rbase = smem_u32(Rs);
#pragma unroll
      for (int kk = 0; kk < kRT / 16; ++kk) {
        uint32_t af[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int i = lane;
          const int row = mt * 16 + (i & 7) + ((i >> 3) & 1) * 8;
          const int ch = kk * 2 + (i >> 4);
          ldsm_x4(pbase + ptile_off(row, ch), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
        }
#pragma unroll
        for (int c = 0; c < NTD; c += 2) {
          uint32_t b0, b1, b2, b3;
          const int i = lane;
          const int row = kk * 16 + (i & 7) + ((i >> 3) & 1) * 8;
          const int ch = (dcol0 >> 3) + c + (i >> 4);
          if (NTD >= 2) {
            ldsm_x4_t(rbase + tile_off<D>(row, ch), b0, b1, b2, b3);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (kSplitFmt && !warp_rope) {
              mma_f16(oacc[mt][c], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
              mma_f16(oacc[mt][c + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b2, b3);
            } else {
              mma_bf16(oacc[mt][c], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
              mma_bf16(oacc[mt][c + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b2, b3);
            }
          }
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- epilogue
  const float oscale = (kSplitFmt && !warp_rope) ? (1.0f / kP2Scale) : 1.0f;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int hl = mt * 16 + g + hh * 8;
      const int h = h0 + hl;
      if (h >= H) continue;
      const float l = lrow[hl], mm = mrow[hl];
      if (p.splits == 1) {
        const float inv = oscale * softmax_norm(mm, l, p.sink, h).f;
        __nv_bfloat16* o = p.out + ((long long)q * H + h) * D + dcol0;
#pragma unroll
        for (int c = 0; c < NTD; ++c) {
          const __nv_bfloat162 v = __floats2bfloat162_rn(oacc[mt][c][2 * hh] * inv, oacc[mt][c][2 * hh + 1] * inv);
          *reinterpret_cast<__nv_bfloat162*>(o + c * 8 + 2 * t4) = v;
        }
        if (p.out_lse != nullptr && warp == 0 && t4 == 0)
          p.out_lse[(long long)q * H + h] = softmax_norm(mm, l, p.sink, h).lse2 * 0.69314718055994531f;
      } else {
        float* o = p.ws_o + (((long long)q * H + h) * p.splits + split) * D + dcol0;
#pragma unroll
        for (int c = 0; c < NTD; ++c) {
          *reinterpret_cast<float2*>(o + c * 8 + 2 * t4) =
              make_float2(oacc[mt][c][2 * hh] * oscale, oacc[mt][c][2 * hh + 1] * oscale);
        }
        if (warp == 0 && t4 == 0) {
          float* ml = p.ws_ml + (((long long)q * H + h) * p.splits + split) * 2;
          ml[0] = mm;
          ml[1] = l;
        }
      }
    }
  }
}

// grid (total_new, heads), block D/4 threads: combine the split partials of one (query, head).
template <int D>
__global__ void __launch_bounds__(D / 4) attend_combine_kernel(AttendParams p) {
  const int q = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int H = p.heads, S = p.splits;
  const float* ml = p.ws_ml + ((long long)q * H + h) * S * 2;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (ml[2 * s + 1] > 0.0f) M = fmaxf(M, ml[2 * s]);
  float Lsum = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < S; ++s) {
    const float l = ml[2 * s + 1];
    if (!(l > 0.0f)) continue;
    const float wgt = exp2f(ml[2 * s] - M);
    Lsum += l * wgt;
    float4 v;
    const long long off = (((long long)q * H + h) * S + s) * D + tid * 4;
    if (p.ws_ob != nullptr) {
      const uint2 raw = *reinterpret_cast<const uint2*>(p.ws_ob + off);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      v = make_float4(a.x, a.y, c.x, c.y);
    } else {
      v = *reinterpret_cast<const float4*>(p.ws_o + off);
    }
    acc.x = fmaf(v.x, wgt, acc.x);
    acc.y = fmaf(v.y, wgt, acc.y);
    acc.z = fmaf(v.z, wgt, acc.z);
    acc.w = fmaf(v.w, wgt, acc.w);
  }
  const SoftmaxNorm nm = softmax_norm(M, Lsum, p.sink, h);
  const float inv = nm.f;
  __nv_bfloat16* o = p.out + ((long long)q * H + h) * D + tid * 4;
  *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  if (tid == 0 && p.out_lse != nullptr)
    p.out_lse[(long long)q * H + h] = nm.lse2 * 0.69314718055994531f;
}

// ----------------------------------------------------------------------------------------------
// launch
// ----------------------------------------------------------------------------------------------

template <int D, int FMT, int MT, bool SV>
static cudaError_t launch_attend_t(const AttendParams& p, int total_new, cudaStream_t st) {
  using L = AttendSmem<D, FMT, MT, SV>;
  static_assert(L::kBytes <= 227 * 1024, "shared memory of one CTA");
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    return cudaFuncSetAttribute(attend_kernel<D, FMT, MT, SV>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  });
  if (ea != cudaSuccess) return ea;
  const int hgroups = (p.heads + L::HG - 1) / L::HG;
  dim3 grid(total_new, hgroups, p.splits);
  attend_kernel<D, FMT, MT, SV><<<grid, 256, L::kBytes, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  attend_combine_kernel<D><<<dim3(total_new, p.heads), D / 4, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attend_combine(const AttendParams& p, int total_new, int D, cudaStream_t st) {
  if (D == 512) attend_combine_kernel<512><<<dim3(total_new, p.heads), 512 / 4, 0, st>>>(p);
  else attend_combine_kernel<128><<<dim3(total_new, p.heads), 128 / 4, 0, st>>>(p);
  return cudaGetLastError();
}

size_t attend_smem_bytes(int D, int fmt, int heads) {
  const bool small = heads <= 16;
  if (D == 512) return small ? AttendSmem<512, LCS_ROW_FP8_SPLIT, 1>::kBytes : AttendSmem<512, LCS_ROW_FP8_SPLIT, 4>::kBytes;
  if (fmt == LCS_ROW_BF16) return small ? AttendSmem<128, LCS_ROW_BF16, 1>::kBytes : AttendSmem<128, LCS_ROW_BF16, 4>::kBytes;
  return small ? AttendSmem<128, LCS_ROW_FP8_SPLIT, 1>::kBytes : AttendSmem<128, LCS_ROW_FP8_SPLIT, 4>::kBytes;
}

template <bool SV>
static cudaError_t launch_attend_sv(const AttendParams& p, int D, int fmt, int total_new, cudaStream_t st) {
  const bool small = p.heads <= 16;
  if (D == 512) {
    if (small) return launch_attend_t<512, LCS_ROW_FP8_SPLIT, 1, SV>(p, total_new, st);
    return launch_attend_t<512, LCS_ROW_FP8_SPLIT, 4, SV>(p, total_new, st);
  }
  if (fmt == LCS_ROW_BF16) {
    if (small) return launch_attend_t<128, LCS_ROW_BF16, 1, SV>(p, total_new, st);
    return launch_attend_t<128, LCS_ROW_BF16, 4, SV>(p, total_new, st);
  }
  if (small) return launch_attend_t<128, LCS_ROW_FP8_SPLIT, 1, SV>(p, total_new, st);
  return launch_attend_t<128, LCS_ROW_FP8_SPLIT, 4, SV>(p, total_new, st);
}

cudaError_t launch_attend(const AttendParams& p, int D, int fmt, int total_new, cudaStream_t st) {
  if (total_new == 0) return cudaSuccess;
  if (p.tc) return launch_attend_tc(p, total_new, st);
  return p.sv ? launch_attend_sv<true>(p, D, fmt, total_new, st) : launch_attend_sv<false>(p, D, fmt, total_new, st);
}

}  // namespace lcsa
