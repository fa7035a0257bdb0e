// Shared-KV multi-query attention on the tcgen05 tensor cores, one 128-row tile per CTA: the
// variant for plans whose splits hold a single tile (short row lists spread over many CTAs, as in
// CSA decode).  It keeps the whole tile in flight at once and transposes the logits through the
// query buffer for the softmax, which a single tile allows; attend_tc.cu holds the multi-tile
// kernel for longer runs.
//
// Defined by: m.x-techcon.com/article/133366, section 2, CSA step 3 (the selected compressed
// entries and the most recent 128 uncompressed tokens are attended together, shared-KV
// multi-query attention) and the HCA paragraph; the efficiency paragraph fixes the row storage
// (RoPE dims BF16, the rest FP8).  Same result as the warp-MMA kernel in attend.cu.
//
// Work of a CTA (query q, 64-head group, tile of rows).  Everything runs in F16 on the rows
// rescaled by their own FP8 scale s_r: R'_r = [rope_r / s_r | codes_r] (the E4M3 codes are exact
// in F16), so that q . row_r = s_r * (q . R'_r) and sum_r p_r row_r = sum_r (p_r s_r) R'_r.
//   gather   row descriptors (top-k entries, window rows); every thread then loads the row
//            scales, its 16-byte pieces of FP8 codes and RoPE dims straight into
//            registers and writes them widened to F16 into the tile: eight K-major chunks of
//            [128 rows][64 dims] (chunk 0 the RoPE dims times 1/s_r); the query arrives by
//            cp.async into eight K-major chunks of [64 heads][64 dims] and becomes F16 in place;
//   S'^T     = R' . Q^T: 32 MMAs (M = 128 rows, N = 64 heads, K = 16), issued back to back;
//   softmax  S'^T is read from tensor memory, scaled by s_r (logit = s_r * S'), transposed
//            through shared memory (over the query buffer); four threads per head take the max
//            and the exponentials (base 2, fp32) over the tile's rows; P' = p * s_r * 2^8 (F16)
//            is written as the K-major [64 heads x 128 rows] operand;
//   O^T      = R'^T . P'^T: 32 MMAs, M = 128 dims per block (the same tile chunks read as an
//            MN-major operand: two 64-dim chunks 16 KB apart, 8-row groups 1024 B apart), N = 64
//            heads, K = 16 rows;
//   epilogue O^T is read from tensor memory (lane = dim, column = head), transposed per warp
//            through shared memory and written in 16-byte pieces, normalised by 2^8 * sum p (one
//            split) or as a BF16 partial with its (max, sum) for the combine kernel.
// Operand chunks use the 128-byte swizzle (16-byte piece j of row r at position j ^ (r % 8)).
// Range: query values within F16 range and row scales below 256 (|x| < 114688), as for the
// warp-MMA kernel.
#include "kernels.cuh"
#include "sm100.cuh"

namespace lcsa {

namespace {

constexpr int kTileRows = 128;
constexpr int kHeads = 64;                // N of both products
constexpr int kD = 512;
constexpr int kNopeBytes = kD - kRope;    // 448 FP8 codes per row
constexpr int kChunk = 16384;             // [128 rows][64 dims] BF16
constexpr int kQChunk = 8192;             // [64 heads][64 dims] BF16
constexpr int kThreads = 256;

struct TcAttSmem {
  static constexpr int kQ = 0;                              // 8 x 8 KB; later the transposes
  static constexpr int kT = kQ + 8 * kQChunk;               // 8 x 16 KB row tile (chunk 0: RoPE)
  static constexpr int kP = kT + 8 * kChunk;                // 2 x 8 KB ([64 heads][64 rows])
  static constexpr int kScale = kP + 2 * kQChunk;           // f32 [128]
  static constexpr int kRinv = kScale + kTileRows * 4;      // f32 [128]  1 / s_r
  static constexpr int kDesc = kRinv + kTileRows * 4;       // long long [128]
  static constexpr int kM = kDesc + kTileRows * 8;          // f32 [64]
  static constexpr int kL = kM + kHeads * 4;                // f32 [64]
  static constexpr int kInv = kL + kHeads * 4;              // f32 [64] output factor per head
  static constexpr int kBar = kInv + kHeads * 4;            // u64 s, pv, drain
  static constexpr int kMisc = kBar + 24;                   // tmem base
  static constexpr int kBytes = kMisc + 16 + 1024;
};
static_assert(TcAttSmem::kBytes <= 227 * 1024, "shared memory");
static_assert(TcAttSmem::kQ % 1024 == 0 && TcAttSmem::kT % 1024 == 0 && TcAttSmem::kP % 1024 == 0,
              "operand chunks on 1024-byte swizzle atoms");
static_assert(kTileRows * 65 * 4 <= 8 * kQChunk, "softmax transpose fits the query buffer");

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

// grid: (total_new, head groups, splits), rows_per_split == 128; with window_split, splits
// 0 .. entry_splits-1 take the entries, split entry_splits the window (part 1: that split alone,
// part 2: the entry splits); otherwise one list of entries then window.
__global__ void __launch_bounds__(kThreads, 1) attend_tc1_kernel(AttendParams p) {
  using L = TcAttSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.x, hg = blockIdx.y;
  const int H = p.heads;
  const int h0 = hg * kHeads;
  const int split = p.part == 1 ? p.entry_splits : blockIdx.z;
  const int32_t* sel = p.topk_idx != nullptr ? p.topk_idx + (long long)q * p.k : nullptr;
  // ---- what does not depend on the indexer first (launched as its programmatic dependent, this
  //      part runs while the indexer's last CTAs merge): the query by cp.async into eight K-major
  //      chunks, the sequence of query q (the row tile's space is free until the rows arrive), its
  //      block-table row head into L2
  for (int idx = tid; idx < kHeads * 64; idx += kThreads) {
    const int h = idx >> 6, c = (idx >> 3) & 7, j = idx & 7;   // head, 64-dim chunk, 16-byte piece
    const bool ok = h0 + h < H;
    const __nv_bfloat16* g = p.q + ((long long)q * H + (ok ? h0 + h : 0)) * kD + c * 64 + j * 8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sbase + L::kQ + c * kQChunk + h * 128 +
                                                                      ((j ^ (h & 7)) << 4)),
                 "l"(g), "r"(ok ? 16 : 0) : "memory");
  }
  cp_async_commit();
  int b;
  const SeqSpan sp = find_seq_span(p.cu_new, p.seq_len, p.num_seqs, q, reinterpret_cast<int*>(smem + L::kT), 8 * kChunk / 4 - 1, &b);
  for (int i = tid * 32; i < p.paging.max_blocks; i += kThreads * 32)
    prefetch_l2(p.paging.table + (long long)b * p.paging.max_blocks + i);
  // ---- the top-k count and the entry indices of this thread's row of the first tiles (written
  //      by the indexer)
  grid_dependency_wait();
  const int spec_r = p.window_split ? (split < p.entry_splits ? split * p.rows_per_split + tid : -1)
                                    : split * p.rows_per_split + tid;
  int spec_j = -1;
  if (sel != nullptr && p.part != 1 && spec_r >= 0 && spec_r < p.k && tid < 2 * kTileRows) spec_j = __ldcg(sel + spec_r);
  const int cnt_g = (sel != nullptr && p.part != 1 && p.topk_cnt != nullptr) ? __ldcg(p.topk_cnt + q) : 0;
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
    while (cnt < p.k && __ldcg(sel + cnt) >= 0) ++cnt;
  }
  const int nvis = (t + 1) / p.m;
  const int W = min(t + 1, kWindow);
  const int R = cnt + W;
  // splits 0 .. entry_splits-1 cover the entries in 128-row tiles, split entry_splits the window
  int r_begin, r_end;
  if (p.window_split) {
    r_begin = split < p.entry_splits ? split * kTileRows : cnt;
    r_end = split < p.entry_splits ? min(cnt, r_begin + kTileRows) : R;
  } else {
    r_begin = split * kTileRows;
    r_end = min(R, r_begin + kTileRows);
  }
  if (r_begin >= r_end) {
    if (p.splits > 1)
      for (int h = tid; h < kHeads; h += kThreads)
        if (h0 + h < H) {
          float* ml = p.ws_ml + (((long long)q * H + h0 + h) * p.splits + split) * 2;
          ml[0] = -INFINITY;
          ml[1] = 0.0f;
        }
    cp_async_wait<0>();   // the query's copies land before the CTA leaves
    return;
  }
  const int nrows = r_end - r_begin;

  long long* desc = reinterpret_cast<long long*>(smem + L::kDesc);
  float* sscale = reinterpret_cast<float*>(smem + L::kScale);
  float* rinv = reinterpret_cast<float*>(smem + L::kRinv);
  float* mrow = reinterpret_cast<float*>(smem + L::kM);
  float* lrow = reinterpret_cast<float*>(smem + L::kL);
  const uint32_t bar_s = sbase + L::kBar;
  const uint32_t bar_pv = bar_s + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);

  // ---- row descriptors and scales: bits 60..61 select the row set (0 entries, 1 new rows,
  //      2 ring), -1 = none
  if (tid < kTileRows) {
    const int r = r_begin + tid;
    long long d = -1;
    if (r < r_end) {
      if (r < cnt) {
        const int j = sel != nullptr ? (r == spec_r ? spec_j : __ldcg(sel + r)) : r;
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
    desc[tid] = d;
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_pv, 1);
    mbar_init(bar_pv + 8, 1);   // drain
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(sbase + L::kMisc, 512);
  __syncthreads();

  // ---- rows: FP8 codes (8 bytes = 8 dims per piece, 56 pieces a row) and RoPE dims (8 per
  //      piece, 8 pieces a row) into registers, then widened into the tile
  {
    constexpr int kNP = kTileRows * 28 / kThreads;     // 14 code pieces (16 FP8 codes) per thread
    constexpr int kRP = kTileRows * 8 / kThreads;      // 4 RoPE pieces per thread
    uint4 cv[kNP];
    uint4 rv[kRP];
    float sc = 0.0f;                                   // threads 0-127: the scale of row tid
    if (tid < kTileRows && desc[tid] >= 0) {
      const long long d = desc[tid];
      const int kind = (int)(d >> 60);
      const long long rw = d & ((1ll << 60) - 1);
      sc = __ldg((kind == 1 ? p.new_rows.scale : (kind == 2 ? p.window.scale : p.entries.scale)) + rw);
    }
#pragma unroll
    for (int it = 0; it < kNP; ++it) {
      const int idx = it * kThreads + tid, r = idx / 28, u = idx % 28;
      const long long d = desc[r];
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
      const long long d = desc[r];
      rv[it] = make_uint4(0u, 0u, 0u, 0u);
      if (d >= 0) {
        const int kind = (int)(d >> 60);
        const long long rw = d & ((1ll << 60) - 1);
        const __nv_bfloat16* src = (kind == 1 ? p.new_rows.rope : (kind == 2 ? p.window.rope : p.entries.rope));
        rv[it] = __ldg(reinterpret_cast<const uint4*>(src + rw * kRope + j * 8));
      }
    }
    if (tid < kTileRows) {
      float s_r = sc;
      if (desc[tid] >= 0 && !(s_r < kMaxRowScale)) {   // p * s_r * 2^8 would leave the f16 range
        report(p.status, LCS_ERR_DEVICE_GUARD);
        desc[tid] = -1;
        s_r = 0.0f;
      }
      sscale[tid] = s_r;
      rinv[tid] = s_r > 0.0f ? __frcp_rn(s_r) : 0.0f;
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
      uint4 h = bf16x8_to_f16x8(rv[it], rinv[r]);
      if (f16x8_nonfinite(h)) {   // |rope| / s_r beyond the f16 range: the row is left out
        report(p.status, LCS_ERR_DEVICE_GUARD);
        desc[r] = -1;
        h = make_uint4(0u, 0u, 0u, 0u);
      }
      *reinterpret_cast<uint4*>(smem + L::kT + r * 128 + ((j ^ (r & 7)) << 4)) = h;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  for (int idx = tid; idx < kHeads * 64; idx += kThreads) {   // query -> F16 in place
    uint4* pc = reinterpret_cast<uint4*>(smem + L::kQ + idx * 16);
    *pc = bf16x8_to_f16x8(*pc, 1.0f);
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem;             // S'^T: columns 0..63
  const uint32_t tm_o = tmem + 64;        // O^T block mb: columns 64 + 64*mb

  constexpr uint32_t kIdS = idesc_f16(0, 128, kHeads);                 // F16, K-major A and B
  constexpr uint32_t kIdO = idesc_f16(0, 128, kHeads) | (1u << 15);    // A (rows^T) MN-major

  // ---- S'^T = R' . Q^T: 8 chunks x 4 steps of 16 dims
  if (tid == 0) {
    tc_fence_after_sync();
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
  bool ok = mbar_wait(bar_s, 0, p.status, nullptr, p.wait_polls);
  ok = __syncthreads_and(ok);
  tc_fence_after_sync();

  // ---- softmax over the tile's rows, per head (transpose through the query buffer)
  float* st = reinterpret_cast<float*>(smem + L::kQ);
  if (ok && warp < 4) {
    const int r = warp * 32 + lane;
    const bool valid = r < nrows && desc[r] >= 0;
    const float lsc = sscale[r] * p.scale_log2;   // logit = s_r * S', in base 2
    uint32_t v[kHeads / 16][16];   // the four loads in flight together, one wait
#pragma unroll
    for (int c16 = 0; c16 < kHeads / 16; ++c16) tmem_ld16(tm_s + ((uint32_t)(warp * 32) << 16) + c16 * 16, v[c16]);
    tmem_ld_wait();
#pragma unroll
    for (int c16 = 0; c16 < kHeads / 16; ++c16)
#pragma unroll
      for (int j = 0; j < 16; ++j) st[r * 65 + c16 * 16 + j] = valid ? __uint_as_float(v[c16][j]) * lsc : -INFINITY;
  }
  __syncthreads();
  {
    const int h = tid >> 2, u = tid & 3;     // four threads per head, 32 rows each
    float mx = -INFINITY;
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, st[(u * 32 + i) * 65 + h]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float sum = 0.0f;
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
      uint4 pk;
      uint32_t* w = &pk.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r0 = u * 32 + g8 * 8 + 2 * e;
        const float a0 = mx == -INFINITY ? 0.0f : exp2f(st[r0 * 65 + h] - mx);
        const float a1 = mx == -INFINITY ? 0.0f : exp2f(st[(r0 + 1) * 65 + h] - mx);
        sum += a0 + a1;
        const __half2 pp = __floats2half2_rn(a0 * sscale[r0] * kP2Scale, a1 * sscale[r0 + 1] * kP2Scale);
        w[e] = *reinterpret_cast<const uint32_t*>(&pp);
      }
      const int rr = u * 32 + g8 * 8;          // first row of this 8-row piece
      const int pc = rr >> 6, j = (rr & 63) >> 3;
      *reinterpret_cast<uint4*>(smem + L::kP + pc * kQChunk + h * 128 + ((j ^ (h & 7)) << 4)) = pk;
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (u == 0) {
      mrow[h] = mx;
      lrow[h] = sum;
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  // ---- O^T = R'^T . P'^T: four 128-dim blocks x 8 steps of 16 rows
  if (tid == 0 && ok) {
    tc_fence_after_sync();
    const uint64_t da = desc_mn_sw128(sbase + L::kT, kChunk, 1024), db = smem_desc_sw128(sbase + L::kP);
#pragma unroll
    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_f16(tm_o + 64 * mb, da + (uint64_t)((2 * mb * kChunk + kk * 2048) >> 4),
                   db + (uint64_t)(((kk >> 2) * kQChunk) >> 4) + 2 * (kk & 3), kIdO, kk > 0 ? 1u : 0u);
    tc_commit(bar_pv);
  }
  if (ok) ok = mbar_wait(bar_pv, 0, p.status, nullptr, p.wait_polls);
  ok = __syncthreads_and(ok);
  tc_fence_after_sync();

  // ---- epilogue: warp w reads lanes 32*(w%4) (dims) of blocks 2*(w/4), 2*(w/4)+1 and writes each
  //      head's 32 dims straight from the registers (64 contiguous bytes a warp and head)
  float* inv_s = reinterpret_cast<float*>(smem + L::kInv);
  for (int h = tid; h < kHeads; h += kThreads)
    inv_s[h] = p.splits == 1 ? softmax_norm(mrow[h], lrow[h], h0 + h < H ? p.sink : nullptr, h0 + h).f / kP2Scale
                             : 1.0f / kP2Scale;
  __syncthreads();
  if (ok) {
    const int quad = warp & 3;
    __nv_bfloat16* base = p.splits == 1 ? p.out + (long long)q * H * kD : p.ws_ob + (long long)q * H * p.splits * kD;
    const long long hstride = p.splits == 1 ? kD : (long long)p.splits * kD;   // between heads
    const long long soff = p.splits == 1 ? 0 : (long long)split * kD;
    const int hn = min(kHeads, H - h0);   // heads of this group that exist
    for (int bi = 0; bi < 2; ++bi) {
      const int mb = 2 * (warp >> 2) + bi;
      __nv_bfloat16* o = base + (long long)h0 * hstride + soff + mb * 128 + quad * 32 + lane;
#pragma unroll 1
      for (int c2 = 0; c2 < kHeads / 32; ++c2) {   // 32 heads: two loads in flight, one wait
        uint32_t v[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tmem_ld16(tm_o + 64 * mb + ((uint32_t)(quad * 32) << 16) + (2 * c2 + c) * 16, v[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int h = (2 * c2 + c) * 16 + j;
            if (h < hn) o[h * hstride] = __float2bfloat16_rn(__uint_as_float(v[c][j]) * inv_s[h]);
          }
      }
    }
    for (int h = tid; h < kHeads; h += kThreads) {
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
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_attend_tc1(const AttendParams& p, int total_new, cudaStream_t st) {
  static PerDeviceOnce attr;
  cudaError_t ea = once_per_device(attr, [] {
    return cudaFuncSetAttribute(attend_tc1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcAttSmem::kBytes);
  });
  if (ea != cudaSuccess) return ea;
  const int z = p.part == 1 ? 1 : (p.part == 2 ? p.entry_splits : p.splits);
  // CSA calls start as programmatic dependents of the preceding kernel in the stream (the
  // indexer lets them start once its scan is done): the kernel reads nothing that kernel writes
  // before grid_dependency_wait()
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(total_new, (p.heads + kHeads - 1) / kHeads, z);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = TcAttSmem::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl;
  cfg.numAttrs = p.topk_idx != nullptr && p.part != 1 ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attend_tc1_kernel, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1 || p.part == 1) return e;
  return launch_attend_combine(p, total_new, kD, st);
}

}  // namespace lcsa
