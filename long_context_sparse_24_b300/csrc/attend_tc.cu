// Shared-KV multi-query attention on the tcgen05 tensor cores for FP8-split rows of D = 512 and
// up to 64 query heads: a CTA takes one query, one 64-head group and a run of 128-row tiles of its
// row list (CSA: top-k entries, then the window; HCA: every visible entry, then the window).
// Plans with one tile per CTA go to the single-tile kernel in attend_tc1.cu.
//
// Defined by: m.x-techcon.com/article/133366, section 2, CSA step 3 (the selected compressed
// entries and the most recent 128 uncompressed tokens are attended together, shared-KV
// multi-query attention) and the HCA paragraph (dense attention over every entry plus the same
// window); the efficiency paragraph fixes the row storage (RoPE dims BF16, the rest FP8).  Same
// result as the warp-MMA kernel in attend.cu: one softmax per head over the rows, o = sum p * row,
// with the row as key and value.
//
// Everything runs in F16 on the rows rescaled by their own FP8 scale s_r:
// R'_r = [rope_r / s_r | codes_r] (the E4M3 codes are exact in F16), so that
// q . row_r = s_r * (q . R'_r) and sum_r p_r row_r = sum_r (p_r s_r) R'_r.  Per tile:
//   gather   row descriptors (warps 4-7, two tiles ahead) and the rows' scales, FP8 codes and
//            RoPE dims loaded into registers one tile ahead (issued right after the current tile
//            is widened, they fly while it computes), then widened to F16 into eight K-major
//            chunks of [128 rows][64 dims]; the
//            query arrives once by cp.async into eight K-major chunks and becomes F16 in place;
//   S'^T     = R' . Q^T: 32 MMAs (M = 128 rows, N = 64 heads, K = 16);
//   softmax  warps 0-3 read S'^T from tensor memory (lane = row), logit = s_r * S'; per-head max
//            and sum over the tile's rows by warp-shuffle reduce-scatters (each lane ends with
//            two heads) and a four-warp combine; exact online softmax: when a head's running max
//            grows, warps 4-7 rescale its O^T columns in tensor memory; P' = p * s_r * 2^8 (F16)
//            is written as the K-major [64 heads x 128 rows] operand;
//   O^T     += R'^T . P'^T: 32 MMAs, M = 128 dims per block (the same tile chunks read as an
//            MN-major operand: two 64-dim chunks 16 KB apart, 8-row groups 1024 B apart), N = 64
//            heads, K = 16 rows.
// Epilogue: O^T read from tensor memory (lane = dim, column = head), transposed per warp through
// shared memory, written in 16-byte pieces normalised by 2^8 * sum p (one split) or as a BF16
// partial with its (max, sum) for the combine kernel.
// Operand chunks use the 128-byte swizzle (16-byte piece j of row r at position j ^ (r % 8)).
// Range: query values within F16 range and row scales below 256 (|x| < 114688), as for the
// warp-MMA kernel.
#include "kernels.cuh"
#include "sm100.cuh"

namespace lcsa {

namespace {

constexpr int kTileRows = 128;
constexpr int kD = 512;
constexpr int kNopeBytes = kD - kRope;    // 448 FP8 codes per row
constexpr int kChunk = 16384;             // [128 rows][64 dims] BF16
constexpr int kThreads = 256;

// HG query heads per CTA (the N of both products): 64, or 16 when a batch has too few queries to
// fill the GPU with 64-head groups (CSA decode).
template <int HG>
struct TcAttSmem {
  static constexpr int kQChunk = HG * 128;                  // [HG heads][64 dims] BF16
  static constexpr int kQ = 0;                              // 8 chunks; the epilogue transposes after the last tile
  static constexpr int kT = kQ + 8 * kQChunk;               // 8 x 16 KB row tile (chunk 0: RoPE)
  static constexpr int kP = kT + 8 * kChunk;                // 2 chunks ([HG heads][64 rows])
  static constexpr int kScale = kP + 2 * kQChunk;           // f32 [2][128]   (tile parity)
  static constexpr int kRinv = kScale + 2 * kTileRows * 4;  // f32 [2][128]   1 / s_r
  // row descriptors: 64 heads, a ring of three tiles (t, t+1, t+2) resolved two tiles ahead; 16
  // heads (shared memory to spare), every tile of the CTA's rows resolved up front
  static constexpr int kDescTiles = 3;                       // ring of three tiles' descriptors
  static constexpr int kDesc = kRinv + 2 * kTileRows * 4;   // long long [kDescTiles][128]
  static constexpr int kRed = kDesc + kDescTiles * kTileRows * 8;   // f32 [4 warps][HG] per-head partials
  static constexpr int kM = kRed + 4 * HG * 4;              // f32 [HG] running max (base 2)
  static constexpr int kL = kM + HG * 4;                    // f32 [HG] running sum
  static constexpr int kMn = kL + HG * 4;                   // f32 [HG] the tile's new max
  static constexpr int kAlpha = kMn + HG * 4;               // f32 [HG] rescale factor of O and l
  static constexpr int kInv = kAlpha + HG * 4;              // f32 [HG] output factor per head
  static constexpr int kBar = kInv + HG * 4;                // u64 s, pv, drain
  static constexpr int kMisc = kBar + 24;                   // tmem base, rescale flag
  static constexpr int kBytes = kMisc + 16 + 1024;
  static constexpr uint32_t kTmemCols = HG == 64 ? 512 : 128;   // S^T (HG) + O^T (4 x HG)
  static_assert(kBytes <= 227 * 1024, "shared memory");
  static_assert(kQ % 1024 == 0 && kT % 1024 == 0 && kP % 1024 == 0, "operand chunks on 1024-byte swizzle atoms");
  static_assert(8 * kQChunk >= 8 * HG * 32 * 4, "epilogue transposes fit the query buffer");
};

// Reduce-scatter of V per-lane values over the 32 lanes of a warp.  Halving rounds (lanes 16, 8,
// ... apart) while a lane holds more than one value, then plain butterfly rounds: afterwards
// v[0 .. max(1, V/32)) hold the reductions of heads scatter_head<V>(lane) + i.
template <int V, bool kMax>
__device__ __forceinline__ void reduce_scatter(float (&v)[V], int lane) {
  constexpr int kHalving = V >= 64 ? 5 : (V == 32 ? 5 : (V == 16 ? 4 : (V == 8 ? 3 : 2)));
#pragma unroll
  for (int r = 0; r < kHalving; ++r) {
    const int off = 16 >> r, n = V >> (r + 1);   // lanes apart, values kept
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = hi ? v[n + i] : v[i];
      const float give = hi ? v[i] : v[n + i];
      const float o = __shfl_xor_sync(0xffffffffu, give, off);
      v[i] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
#pragma unroll
  for (int off = 16 >> kHalving; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v[0], off);
    v[0] = kMax ? fmaxf(v[0], o) : v[0] + o;
  }
}

// First head of a lane's values after reduce_scatter<V> (lane bit 4 selects the upper half of the
// values in the first round, bit 3 in the second, ...).
template <int V>
__device__ __forceinline__ int scatter_head(int lane) {
  constexpr int kHalving = V >= 64 ? 5 : (V == 32 ? 5 : (V == 16 ? 4 : (V == 8 ? 3 : 2)));
  int h = 0;
#pragma unroll
  for (int r = 0; r < kHalving; ++r)
    if (lane & (16 >> r)) h += V >> (r + 1);
  return h;
}

// Whether a lane writes its reduced values (lanes that differ only in the butterfly bits hold
// copies).
template <int V>
__device__ __forceinline__ bool scatter_writer(int lane) {
  constexpr int kHalving = V >= 64 ? 5 : (V == 32 ? 5 : (V == 16 ? 4 : (V == 8 ? 3 : 2)));
  return (lane & ((16 >> kHalving) * 2 - 1)) == 0 || kHalving == 5;
}

__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

constexpr float kP2Scale = 256.0f;   // power-of-two pre-scale of p * s_r for the F16 operand

// 8 FP8 codes -> 8 F16 (one 16-byte operand piece), exact.
__device__ __forceinline__ uint4 widen8(uint2 codes) {
  uint4 o;
  o.x = e4m3x2_to_f16x2((uint16_t)(codes.x & 0xFFFF));
  o.y = e4m3x2_to_f16x2((uint16_t)(codes.x >> 16));
  o.z = e4m3x2_to_f16x2((uint16_t)(codes.y & 0xFFFF));
  o.w = e4m3x2_to_f16x2((uint16_t)(codes.y >> 16));
  return o;
}

// 16 FP8 codes -> two pieces of 8 F16, exact.
__device__ __forceinline__ void widen16(uint4 codes, uint4& lo, uint4& hi) {
  lo = widen8(make_uint2(codes.x, codes.y));
  hi = widen8(make_uint2(codes.z, codes.w));
}

// 8 BF16 -> 8 F16, each multiplied by m (m = 1: exact conversion within the F16 range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float m) {
  uint32_t* w = &v.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    const __half2 h = __floats2half2_rn(f.x * m, f.y * m);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return v;
}

}  // namespace

// grid: (total_new, head groups, splits); splits 0 .. entry_splits-1 take 128-row tiles of the
// entries, split entry_splits the window rows (part 1: that split alone, part 2: the entry splits).
template <int HG>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(AttendParams p) {
  using L = TcAttSmem<HG>;
  constexpr int kQChunk = L::kQChunk;
  constexpr int HH = HG / 2;                       // heads a warp takes in the logit and P' passes
  constexpr int kVals = HH >= 32 ? HH / 32 : 1;   // per-lane values after a reduce-scatter
  static_assert(HH >= 8 && HH % 16 == 0, "two warps a TMEM lane quadrant, half the heads each");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.x, hg = blockIdx.y;
  const int H = p.heads;
  const int h0 = hg * HG;
  // this CTA's split, and (before the sequence is known) the query's top-k count and the entry
  // indices of the rows of its first tiles, read with the batch's offsets
  const int split = p.part == 1 ? p.entry_splits : blockIdx.z;
  const int32_t* sel = p.topk_idx != nullptr ? p.topk_idx + (long long)q * p.k : nullptr;
  const int spec_r = p.window_split ? (split < p.entry_splits ? split * p.rows_per_split + tid : -1)
                                    : split * p.rows_per_split + tid;   // this thread's row of the first tiles
  int spec_j = -1;
  if (sel != nullptr && p.part != 1 && spec_r >= 0 && spec_r < p.k && tid < 2 * kTileRows) spec_j = __ldg(sel + spec_r);
  const int cnt_g = (sel != nullptr && p.part != 1 && p.topk_cnt != nullptr) ? __ldg(p.topk_cnt + q) : 0;
  // sequence of query q (the row tile's space is free until the rows arrive)
  int b;
  const SeqSpan sp = find_seq_span(p.cu_new, p.seq_len, p.num_seqs, q, reinterpret_cast<int*>(smem + L::kT), 8 * kChunk / 4 - 1, &b);
  // the top-k list and the sequence's block-table row head for L2 while the count is read
  if (p.topk_idx != nullptr && p.part != 1)
    for (int i = tid * 32; i < p.k; i += kThreads * 32) prefetch_l2(p.topk_idx + (long long)q * p.k + i);
  for (int i = tid * 32; i < p.paging.max_blocks; i += kThreads * 32)
    prefetch_l2(p.paging.table + (long long)b * p.paging.max_blocks + i);
  const int n0 = sp.n0();
  const int t = n0 + (q - sp.q0);
  int cnt;
  if (p.part == 1) {
    cnt = 0;                         // window split alone: the entry list is not needed
  } else if (sel == nullptr) {
    cnt = (t + 1) / p.m;             // HCA: every visible entry
  } else if (p.topk_cnt != nullptr) {
    cnt = min(cnt_g, p.k);
  } else {
    cnt = 0;
    while (cnt < p.k && sel[cnt] >= 0) ++cnt;
  }
  const int nvis = (t + 1) / p.m;
  const int W = min(t + 1, kWindow);
  const int R = cnt + W;
  // this CTA's rows: CSA (window apart): splits 0 .. entry_splits-1 cover the entries, split
  // entry_splits the window; HCA: one list of entries then window, rows_per_split each
  int r_begin, r_end;
  if (p.window_split) {
    r_begin = split < p.entry_splits ? split * p.rows_per_split : cnt;
    r_end = split < p.entry_splits ? min(cnt, r_begin + p.rows_per_split) : R;
  } else {
    r_begin = split * p.rows_per_split;
    r_end = min(R, r_begin + p.rows_per_split);
  }
  if (r_begin >= r_end) {
    if (p.splits > 1)
      for (int h = tid; h < HG; h += kThreads)
        if (h0 + h < H) {
          float* ml = p.ws_ml + (((long long)q * H + h0 + h) * p.splits + split) * 2;
          ml[0] = -INFINITY;
          ml[1] = 0.0f;
        }
    return;
  }
  const int ntiles = (r_end - r_begin + kTileRows - 1) / kTileRows;

  long long* desc = reinterpret_cast<long long*>(smem + L::kDesc);
  float* sscale = reinterpret_cast<float*>(smem + L::kScale);
  float* rinv = reinterpret_cast<float*>(smem + L::kRinv);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  float* mrow = reinterpret_cast<float*>(smem + L::kM);
  float* lrow = reinterpret_cast<float*>(smem + L::kL);
  float* mnew = reinterpret_cast<float*>(smem + L::kMn);
  float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);
  const uint32_t bar_s = sbase + L::kBar;
  const uint32_t bar_pv = bar_s + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile int* rescale_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  // ---- the query first (independent of the rows): cp.async into eight K-major chunks
  for (int idx = tid; idx < HG * 64; idx += kThreads) {
    const int h = idx >> 6, c = (idx >> 3) & 7, j = idx & 7;   // head, 64-dim chunk, 16-byte piece
    const bool okq = h0 + h < H;
    const __nv_bfloat16* g = p.q + ((long long)q * H + (okq ? h0 + h : 0)) * kD + c * 64 + j * 8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sbase + L::kQ + c * kQChunk + h * 128 +
                                                                      ((j ^ (h & 7)) << 4)),
                 "l"(g), "r"(okq ? 16 : 0) : "memory");
  }
  cp_async_commit();

  // row descriptor of tile row i of tile tt: bits 60..61 select the row set (0 entries, 1 new rows,
  // 2 ring), -1 = none
  auto make_desc = [&](int tt, int i) -> long long {
    const int r = r_begin + tt * kTileRows + i;
    long long d = -1;
    if (r < r_end) {
      if (r < cnt) {
        const int j = sel != nullptr ? (r == spec_r ? spec_j : sel[r]) : r;
        long long row = -1;
        if (j >= 0 && j < nvis) row = entry_row(p.paging, b, j, p.entries.num_rows);
        if (row < 0) report(p.status, LCS_ERR_DEVICE_GUARD);
        d = row;
      } else {
        const int pos = t - W + 1 + (r - cnt);
        if (pos >= n0 && p.new_rows.nope != nullptr) {
          const long long row = (long long)sp.q0 + (pos - n0);
          d = row < p.new_rows.num_rows ? (row | (1ll << 60)) : -1;
        } else {
          const long long row = (long long)b * kWindow + (pos % kWindow);
          d = row < p.window.num_rows ? (row | (2ll << 60)) : -1;
        }
        if (d < 0) report(p.status, LCS_ERR_DEVICE_GUARD);
      }
    }
    return d;
  };

  constexpr int kNP = kTileRows * 28 / kThreads;     // 14 code pieces (16 FP8 codes) per thread
  constexpr int kRP = kTileRows * 8 / kThreads;      // 4 RoPE pieces (8 BF16) per thread
  uint4 cv[kNP];
  uint4 rv[kRP];
  float sc = 0.0f;                                   // threads 0-127: the scale of row tid
  auto dslot = [&](int tt) { return tt % 3; };
  // issue the loads of tile tt (descriptors in desc[dslot(tt)]) into registers
  auto load_tile = [&](int tt) {
    const long long* dd = desc + dslot(tt) * kTileRows;
    sc = 0.0f;
    if (tid < kTileRows && dd[tid] >= 0) {
      const long long d = dd[tid];
      const int kind = (int)(d >> 60);
      const long long rw = d & ((1ll << 60) - 1);
      sc = __ldg((kind == 1 ? p.new_rows.scale : (kind == 2 ? p.window.scale : p.entries.scale)) + rw);
    }
#pragma unroll
    for (int it = 0; it < kNP; ++it) {
      const int idx = it * kThreads + tid, r = idx / 28, u = idx % 28;
      const long long d = dd[r];
      cv[it] = make_uint4(0u, 0u, 0u, 0u);
      if (d >= 0) {
        const int kind = (int)(d >> 60);
        const long long rw = d & ((1ll << 60) - 1);
        const uint8_t* src = (kind == 1 ? p.new_rows.nope : (kind == 2 ? p.window.nope : p.entries.nope));
        cv[it] = __ldg(reinterpret_cast<const uint4*>(src + rw * kNopeBytes + u * 16));
      }
    }
#pragma unroll
    for (int it = 0; it < kRP; ++it) {
      const int idx = it * kThreads + tid, r = idx >> 3, j = idx & 7;
      const long long d = dd[r];
      rv[it] = make_uint4(0u, 0u, 0u, 0u);
      if (d >= 0) {
        const int kind = (int)(d >> 60);
        const long long rw = d & ((1ll << 60) - 1);
        const __nv_bfloat16* src = (kind == 1 ? p.new_rows.rope : (kind == 2 ? p.window.rope : p.entries.rope));
        rv[it] = __ldg(reinterpret_cast<const uint4*>(src + rw * kRope + j * 8));
      }
    }
  };

  if (tid < kTileRows) {
    desc[tid] = make_desc(0, tid);
  } else if (ntiles > 1) {
    desc[tid] = make_desc(1, tid - kTileRows);   // tile 1 in desc[1]
  }
  if (tid < HG) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.0f;
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_pv, 1);
    mbar_init(bar_pv + 8, 1);   // drain
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(sbase + L::kMisc, L::kTmemCols);
  __syncthreads();
  load_tile(0);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem;             // S'^T: columns 0 .. HG-1
  const uint32_t tm_o = tmem + HG;        // O^T block mb: columns HG + HG*mb

  constexpr uint32_t kIdS = idesc_f16(0, 128, HG);                 // F16, K-major A and B
  constexpr uint32_t kIdO = idesc_f16(0, 128, HG) | (1u << 15);    // A (rows^T) MN-major
  bool ok = true;

  for (int tt = 0; tt < ntiles; ++tt) {
    const int bp = tt & 1;
    const int trows = min(kTileRows, r_end - r_begin - tt * kTileRows);
    // ---- 1. the previous tile's PV MMAs have read the tile buffer and P
    if (tt > 0) ok = mbar_wait(bar_pv, (tt - 1) & 1, p.status, nullptr, p.wait_polls) && ok;
    ok = __syncthreads_and(ok);
    if (!ok) break;
    // ---- 2. this tile's scales, then its rows widened into the tile buffer
    if (tid < kTileRows) {
      float s_r = sc;
      if (desc[dslot(tt) * kTileRows + tid] >= 0 && !(s_r < kMaxRowScale)) {   // p * s_r * 2^8 leaves f16
        report(p.status, LCS_ERR_DEVICE_GUARD);
        desc[dslot(tt) * kTileRows + tid] = -1;
        s_r = 0.0f;
      }
      sscale[bp * kTileRows + tid] = s_r;
      rinv[bp * kTileRows + tid] = s_r > 0.0f ? __frcp_rn(s_r) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kNP; ++it) {
      const int idx = it * kThreads + tid, r = idx / 28, u = idx % 28;
      const int c = 1 + (u >> 2), j = (u & 3) * 2;        // chunk, first 16-byte piece of 8 dims
      uint4 lo, hi;
      widen16(cv[it], lo, hi);
      *reinterpret_cast<uint4*>(smem + L::kT + c * kChunk + r * 128 + ((j ^ (r & 7)) << 4)) = lo;
      *reinterpret_cast<uint4*>(smem + L::kT + c * kChunk + r * 128 + (((j + 1) ^ (r & 7)) << 4)) = hi;
    }
#pragma unroll
    for (int it = 0; it < kRP; ++it) {
      const int idx = it * kThreads + tid, r = idx >> 3, j = idx & 7;
      uint4 h = bf16x8_to_f16x8(rv[it], rinv[bp * kTileRows + r]);
      if (f16x8_nonfinite(h)) {   // |rope| / s_r beyond the f16 range: the row is left out
        report(p.status, LCS_ERR_DEVICE_GUARD);
        desc[dslot(tt) * kTileRows + r] = -1;
        h = make_uint4(0u, 0u, 0u, 0u);
      }
      *reinterpret_cast<uint4*>(smem + L::kT + r * 128 + ((j ^ (r & 7)) << 4)) = h;
    }
    // the next tile's rows go out now and fly while this tile computes
    if (tt + 1 < ntiles) load_tile(tt + 1);
    if (tt == 0) {
      cp_async_wait<0>();
      __syncthreads();
      for (int idx = tid; idx < HG * 64; idx += kThreads) {   // query -> F16 in place
        uint4* pc = reinterpret_cast<uint4*>(smem + L::kQ + idx * 16);
        *pc = bf16x8_to_f16x8(*pc, 1.0f);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // ---- 3. S'^T = R' . Q^T
    if (tid == 0) {
      // (descriptors: the base ones plus constant offsets of the start-address field)
      const uint64_t da = smem_desc_sw128(sbase + L::kT), db = smem_desc_sw128(sbase + L::kQ);
#pragma unroll
      for (int c = 0; c < 8; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16(tm_s, da + (uint64_t)((c * kChunk) >> 4) + 2 * kk, db + (uint64_t)((c * kQChunk) >> 4) + 2 * kk,
                     kIdS, (c > 0 || kk > 0) ? 1u : 0u);
      tc_commit(bar_s);
    }
    // ---- 4. logits and the tile max per head: warp w takes the rows of TMEM lane quadrant w % 4
    //      and half of the heads (w / 4); warps 4-7 also build the descriptors of tile tt + 2
    const int quad = warp & 3, hhalf = warp >> 2;
    const int r = quad * 32 + lane;           // tile row
    const int hb = scatter_head<HH>(lane);
    const bool hw_lane = scatter_writer<HH>(lane);
    const bool rvalid = r < trows && desc[dslot(tt) * kTileRows + r] >= 0;
    if (warp >= 4 && tt + 2 < ntiles) desc[((tt + 2) % 3) * kTileRows + tid - 128] = make_desc(tt + 2, tid - 128);
    ok = mbar_wait(bar_s, tt & 1, p.status, nullptr, p.wait_polls) && ok;
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after_sync();
    if (ok) {
      const float lsc = sscale[bp * kTileRows + r] * p.scale_log2;   // logit = s_r * S', base 2
      float w[HH];
      uint32_t u[HH / 16][16];   // every load in flight, one wait
#pragma unroll
      for (int c16 = 0; c16 < HH / 16; ++c16)
        tmem_ld16(tm_s + ((uint32_t)(quad * 32) << 16) + hhalf * HH + c16 * 16, u[c16]);
      tmem_ld_wait();
#pragma unroll
      for (int c16 = 0; c16 < HH / 16; ++c16)
#pragma unroll
        for (int j = 0; j < 16; ++j) w[c16 * 16 + j] = rvalid ? __uint_as_float(u[c16][j]) * lsc : -INFINITY;
      reduce_scatter<HH, true>(w, lane);
      if (hw_lane)
#pragma unroll
        for (int i = 0; i < kVals; ++i) red[quad * HG + hhalf * HH + hb + i] = w[i];
    }
    ok = __syncthreads_and(ok);
    if (!ok) break;
    // ---- 5. new running max and rescale factors per head
    if (tid == 0) *rescale_flag = 0;
    __syncthreads();
    if (tid < HG) {
      const float mt = fmaxf(fmaxf(red[tid], red[HG + tid]), fmaxf(red[2 * HG + tid], red[3 * HG + tid]));
      const float mo = mrow[tid];
      const float mn = fmaxf(mo, mt);
      const float al = (mo == -INFINITY || mn == -INFINITY) ? 0.0f : exp2f(mo - mn);
      mnew[tid] = mn;
      alpha_s[tid] = al;
      if (tt > 0 && al < 1.0f) *rescale_flag = 1;
    }
    __syncthreads();
    // ---- 6. P' and the tile sum per head (warp w: its quadrant's rows, its half of the heads),
    //      then, where the max grew, O^T rescaled (warp w: its quadrant's lanes, blocks of its half)
    {
      float w[HH];
      const float srow = sscale[bp * kTileRows + r] * kP2Scale;
      const float lsc = sscale[bp * kTileRows + r] * p.scale_log2;
      tc_fence_after_sync();
      {   // the logits again, from tensor memory (every load in flight, one wait)
        uint32_t u[HH / 16][16];
#pragma unroll
        for (int c16 = 0; c16 < HH / 16; ++c16)
          tmem_ld16(tm_s + ((uint32_t)(quad * 32) << 16) + hhalf * HH + c16 * 16, u[c16]);
        tmem_ld_wait();
#pragma unroll
        for (int c16 = 0; c16 < HH / 16; ++c16)
#pragma unroll
          for (int j = 0; j < 16; ++j) w[c16 * 16 + j] = rvalid ? __uint_as_float(u[c16][j]) * lsc : -INFINITY;
      }
#pragma unroll
      for (int hl = 0; hl < HH; hl += 2) {
        const int h = hhalf * HH + hl;
        const float m0 = mnew[h], m1 = mnew[h + 1];
        const float a0 = m0 == -INFINITY ? 0.0f : exp2f(w[hl] - m0);
        const float a1 = m1 == -INFINITY ? 0.0f : exp2f(w[hl + 1] - m1);
        w[hl] = a0;
        w[hl + 1] = a1;
        // P'[h][r], [h+1][r]: K-major, chunk r/64, piece (r%64)/8 of head row h, element r%8
        const int pc = r >> 6, pj = (r & 63) >> 3, pe = r & 7;
        *reinterpret_cast<__half*>(smem + L::kP + pc * kQChunk + h * 128 + ((pj ^ (h & 7)) << 4) + pe * 2) =
            __float2half_rn(a0 * srow);
        *reinterpret_cast<__half*>(smem + L::kP + pc * kQChunk + (h + 1) * 128 + ((pj ^ ((h + 1) & 7)) << 4) + pe * 2) =
            __float2half_rn(a1 * srow);
      }
      reduce_scatter<HH, false>(w, lane);
      if (hw_lane)
#pragma unroll
        for (int i = 0; i < kVals; ++i) red[quad * HG + hhalf * HH + hb + i] = w[i];
    }
    if (*rescale_flag) {
#pragma unroll 1
      for (int cc = 0; cc < 2 * (HG / 32); ++cc) {   // two 16-column chunks at a time, one wait
        const int mb = 2 * hhalf + cc / (HG / 32), c0 = (cc % (HG / 32)) * 2;
        uint32_t u[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld16(tm_o + HG * mb + ((uint32_t)(quad * 32) << 16) + (c0 + c) * 16, u[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int j = 0; j < 16; ++j) u[c][j] = __float_as_uint(__uint_as_float(u[c][j]) * alpha_s[(c0 + c) * 16 + j]);
          tmem_st16(tm_o + HG * mb + ((uint32_t)(quad * 32) << 16) + (c0 + c) * 16, u[c]);
        }
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // ---- 7. running statistics; O^T += R'^T . P'^T
    if (tid < HG) {
      lrow[tid] = lrow[tid] * alpha_s[tid] + (red[tid] + red[HG + tid]) + (red[2 * HG + tid] + red[3 * HG + tid]);
      mrow[tid] = mnew[tid];
    }
    if (tid == 0) {
      const uint64_t da = desc_mn_sw128(sbase + L::kT, kChunk, 1024), db = smem_desc_sw128(sbase + L::kP);
#pragma unroll
      for (int mb = 0; mb < 4; ++mb)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 rows per step: two 8-row groups
          tc_mma_f16(tm_o + HG * mb, da + (uint64_t)((2 * mb * kChunk + kk * 2048) >> 4),
                     db + (uint64_t)(((kk >> 2) * kQChunk) >> 4) + 2 * (kk & 3), kIdO, (tt > 0 || kk > 0) ? 1u : 0u);
      tc_commit(bar_pv);
    }
  }
  if (ok) ok = mbar_wait(bar_pv, (ntiles - 1) & 1, p.status, nullptr, p.wait_polls);
  ok = __syncthreads_and(ok);
  tc_fence_after_sync();

  // ---- epilogue: warp w reads lanes 32*(w%4) (dims) of blocks 2*(w/4), 2*(w/4)+1, transposes
  //      them through its own 8 KB of the query buffer and writes 16-byte pieces
  float* inv_s = reinterpret_cast<float*>(smem + L::kInv);
  for (int h = tid; h < HG; h += kThreads)
    inv_s[h] = p.splits == 1 ? softmax_norm(mrow[h], lrow[h], h0 + h < H ? p.sink : nullptr, h0 + h).f / kP2Scale
                             : 1.0f / kP2Scale;
  __syncthreads();
  if (ok) {
    const int quad = warp & 3;
    float* tb = reinterpret_cast<float*>(smem + L::kQ) + warp * (HG * 32);   // [HG heads][32 dims]
    for (int bi = 0; bi < 2; ++bi) {
      const int mb = 2 * (warp >> 2) + bi;
      const int dim0 = mb * 128 + quad * 32;
      uint32_t v[HG / 16][16];   // every load in flight, one wait
#pragma unroll
      for (int c16 = 0; c16 < HG / 16; ++c16)
        tmem_ld16(tm_o + HG * mb + ((uint32_t)(quad * 32) << 16) + c16 * 16, v[c16]);
      tmem_ld_wait();
#pragma unroll
      for (int c16 = 0; c16 < HG / 16; ++c16)
#pragma unroll
        for (int j = 0; j < 16; ++j) tb[(c16 * 16 + j) * 32 + lane] = __uint_as_float(v[c16][j]) * inv_s[c16 * 16 + j];
      __syncwarp();
#pragma unroll 4
      for (int i = 0; i < HG / 4; ++i) {
        const int h = i * 4 + (lane >> 3), d4 = (lane & 7) * 4;
        if (h0 + h < H) {
          const float4 o = *reinterpret_cast<const float4*>(tb + h * 32 + d4);
          if (p.splits == 1) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
            uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
            *reinterpret_cast<uint2*>(p.out + ((long long)q * H + h0 + h) * kD + dim0 + d4) = pk;
          } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
            uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
            *reinterpret_cast<uint2*>(p.ws_ob + (((long long)q * H + h0 + h) * p.splits + split) * kD + dim0 + d4) = pk;
          }
        }
      }
      __syncwarp();
    }
    for (int h = tid; h < HG; h += kThreads) {
      if (h0 + h >= H) continue;
      const float l = lrow[h], mm = mrow[h];
      if (p.splits == 1) {
        if (p.out_lse != nullptr)
          p.out_lse[(long long)q * H + h0 + h] = softmax_norm(mm, l, p.sink, h0 + h).lse2 * 0.69314718055994531f;
      } else {
        float* ml = p.ws_ml + (((long long)q * H + h0 + h) * p.splits + split) * 2;
        ml[0] = mm;
        ml[1] = l;
      }
    }
  }
  // after a wait gave up, the MMAs still in flight complete before tensor memory is released
  if (tid == 0 && !ok) {
    tc_commit(bar_pv + 8);
    mbar_wait(bar_pv + 8, 0, nullptr, nullptr, kWaitPolls);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

namespace {

template <int HG>
cudaError_t launch_attend_tc_t(const AttendParams& p, int total_new, cudaStream_t st) {
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    return cudaFuncSetAttribute(attend_tc_kernel<HG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcAttSmem<HG>::kBytes);
  });
  if (ea != cudaSuccess) return ea;
  const int z = p.part == 1 ? 1 : (p.part == 2 ? p.entry_splits : p.splits);
  dim3 grid(total_new, (p.heads + HG - 1) / HG, z);
  attend_tc_kernel<HG><<<grid, kThreads, TcAttSmem<HG>::kBytes, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1 || p.part == 1) return e;
  return launch_attend_combine(p, total_new, kD, st);
}

}  // namespace

cudaError_t launch_attend_tc(const AttendParams& p, int total_new, cudaStream_t st) {
  if (p.rows_per_split == kTileRows) return launch_attend_tc1(p, total_new, st);   // one tile per CTA
  return launch_attend_tc_t<64>(p, total_new, st);
}

}  // namespace lcsa
