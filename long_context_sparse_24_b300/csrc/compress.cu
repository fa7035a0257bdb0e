// KV compression (CSA m=4 with overlapping windows, HCA m'=128) and the state-cache update.
//
// Defined by: m.x-techcon.com/article/133366, section 2 "核心技术创新：混合压缩注意力", CSA step 1
// (each raw token gets a learned weight plus a positional bias, the weights are softmax-
// normalised and the rows summed with them; adjacent blocks overlap) and the HCA paragraph
// (ratio 128); section 4 "专门为混合注意力设计的KV缓存管理" (state cache holds the window rows and
// the uncompressed tail; the compressed cache is allocated in blocks).  Storage format from the
// same page's efficiency paragraph (RoPE dims BF16, the rest FP8).
//
// Work split: one warp per entry for windows of up to 16 rows (CSA), one CTA of 8 warps per
// entry for longer windows (HCA).  Every raw row is read with 16-byte vector loads; lane l of a
// warp owns the 16-byte chunks l, l+32, ... of a row, so a warp-wide load is one contiguous
// 512-byte segment.  The arithmetic of one entry does not depend on how many entries the call
// completes, so decode-time (one token) and prefill-time (many tokens) compression give the
// same bits.
#include "kernels.cuh"

namespace lcsa {



template <int D>
struct RowChunks {
  static constexpr int kChunks = D / 8;                 // 16-byte chunks of a bf16 row
  static constexpr int kPerLane = (kChunks + 31) / 32;  // chunks owned by one lane
};

// Load lane-owned chunks of a bf16 row as fp32.
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int lane, float (&v)[RowChunks<D>::kPerLane][8]) {
#pragma unroll
  for (int i = 0; i < RowChunks<D>::kPerLane; ++i) {
    int c = lane + 32 * i;
    if (c < RowChunks<D>::kChunks) {
      uint4 u = *reinterpret_cast<const uint4*>(row + c * 8);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f = __bfloat1622float2(h[k]);
        v[i][2 * k] = f.x;
        v[i][2 * k + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[i][k] = 0.0f;
    }
  }
}

// Lane-owned 16-byte chunks of a bf16 row, raw (issue all loads first, convert later).
template <int D>
__device__ __forceinline__ void load_row_raw(const __nv_bfloat16* row, int lane, uint4 (&r)[RowChunks<D>::kPerLane]) {
#pragma unroll
  for (int i = 0; i < RowChunks<D>::kPerLane; ++i) {
    const int c = lane + 32 * i;
    r[i] = c < RowChunks<D>::kChunks ? *reinterpret_cast<const uint4*>(row + c * 8) : make_uint4(0, 0, 0, 0);
  }
}

template <int D>
__device__ __forceinline__ void unpack_row(const uint4 (&r)[RowChunks<D>::kPerLane], int lane,
                                           float (&v)[RowChunks<D>::kPerLane][8]) {
#pragma unroll
  for (int i = 0; i < RowChunks<D>::kPerLane; ++i) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r[i]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      v[i][2 * k] = f.x;
      v[i][2 * k + 1] = f.y;
    }
  }
}

// Quantise one row held by a warp (lane-owned chunks) and store it as row `r` of `dst`.
template <int D>
__device__ __forceinline__ void store_row(const Rows& dst, long long r, int lane,
                                          const float (&v)[RowChunks<D>::kPerLane][8]) {
  constexpr int C = RowChunks<D>::kChunks;
  if (dst.format == LCS_ROW_BF16) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(dst.nope) + r * D;
#pragma unroll
    for (int i = 0; i < RowChunks<D>::kPerLane; ++i) {
      int c = lane + 32 * i;
      if (c < C) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[i][2 * k], v[i][2 * k + 1]);
        *reinterpret_cast<uint4*>(out + c * 8) = u;
      }
    }
    return;
  }
  // FP8 split: chunks 0..7 are the RoPE dims (BF16), chunks 8.. the E4M3 dims.
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < RowChunks<D>::kPerLane; ++i) {
    int c = lane + 32 * i;
    if (c >= kRope / 8 && c < C) {
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[i][k]));
    }
  }
  amax = warp_max(amax);
  const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
#pragma unroll
  for (int i = 0; i < RowChunks<D>::kPerLane; ++i) {
    int c = lane + 32 * i;
    if (c < kRope / 8) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[i][2 * k], v[i][2 * k + 1]);
      *reinterpret_cast<uint4*>(dst.rope + r * kRope + c * 8) = u;
    } else if (c < C) {
      uint2 u;
      uint16_t* q = reinterpret_cast<uint16_t*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        q[k] = f32x2_to_e4m3x2(__fdiv_rn(v[i][2 * k], s), __fdiv_rn(v[i][2 * k + 1], s));
      *reinterpret_cast<uint2*>(dst.nope + r * (D - kRope) + (c - kRope / 8) * 8) = u;
    }
  }
  if (lane == 0) dst.scale[r] = s;
}

// Pointer to raw token t of sequence span sp (t < n0: the pending ring; t >= n0: this call's rows).
__device__ __forceinline__ const __nv_bfloat16* token_row(const CompressParams& p, int b, const SeqSpan& sp,
                                                          int t, int D) {
  if (t >= sp.n0()) return p.raw + (long long)(sp.q0 + t - sp.n0()) * D;
  return p.pending + ((long long)b * p.pending_slots + (t % p.pending_slots)) * D;
}

// grid: (ceil(max_entries_per_call / EPC), num_seqs), block 256.  WPE warps per entry.
template <int D, int WPE>
__global__ void __launch_bounds__(256) compress_entries_kernel(CompressParams p) {
  constexpr int EPC = 8 / WPE;
  constexpr int PL = RowChunks<D>::kPerLane;
  constexpr int kMaxRows = 256;
  __shared__ float zbuf[EPC][kMaxRows];
  __shared__ float red[WPE > 1 ? 8 : 1][WPE > 1 ? D : 1];

  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e_local = warp / WPE, wi = warp % WPE;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int m = p.m;
  const int j_first = sp.n0() / m, j_end = sp.n1 / m;
  const int j = j_first + blockIdx.x * EPC + e_local;
  const bool active = j < j_end;  // warp-uniform; whole entry group shares it
  const int R = p.overlap ? 2 * m : m;
  const int lo = p.overlap ? (j - 1) * m : j * m;

  // phase 1: scores z_t = w . k_t + b[offset]
  float wv[PL][8];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    int c = lane + 32 * i;
#pragma unroll
    for (int k = 0; k < 8; ++k) wv[i][k] = c < RowChunks<D>::kChunks ? p.w[c * 8 + k] : 0.0f;
  }
  if (active) {
    // rows in batches of 4 so that four row loads are in flight per warp
    for (int rb = wi; rb < R; rb += 4 * WPE) {
      uint4 raw[4][PL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rr = rb + u * WPE, t = lo + rr;
        if (rr < R && t >= 0) load_row_raw<D>(token_row(p, b, sp, t, D), lane, raw[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rr = rb + u * WPE, t = lo + rr;
        if (rr >= R) break;
        float z = -INFINITY;
        if (t >= 0) {
          float v[PL][8];
          unpack_row<D>(raw[u], lane, v);
          float acc = 0.0f;
#pragma unroll
          for (int i = 0; i < PL; ++i)
#pragma unroll
            for (int k = 0; k < 8; ++k) acc = fmaf(wv[i][k], v[i][k], acc);
          z = warp_sum(acc) + p.bias[rr];
        }
        if (lane == 0) zbuf[e_local][rr] = z;
      }
    }
  }
  __syncthreads();
  if (!active) return;  // entry groups are whole: no later block-wide barrier is skipped unevenly

  // phase 2: softmax weights over the rows that exist, weighted sum
  float zmax = -INFINITY;
  for (int rr = lane; rr < R; rr += 32) zmax = fmaxf(zmax, zbuf[e_local][rr]);
  zmax = warp_max(zmax);
  float zsum = 0.0f;
  if (R <= 16) {
    // every lane sums in row order: the streaming kernel's order, so that an entry has the same
    // bits whichever kernel forms it
    for (int rr = 0; rr < R; ++rr) {
      const float z = zbuf[e_local][rr];
      zsum += (z == -INFINITY) ? 0.0f : expf(z - zmax);
    }
  } else {
    for (int rr = lane; rr < R; rr += 32) {
      const float z = zbuf[e_local][rr];
      zsum += (z == -INFINITY) ? 0.0f : expf(z - zmax);
    }
    zsum = warp_sum(zsum);
  }
  const float inv = 1.0f / zsum;

  float acc[PL][8];
#pragma unroll
  for (int i = 0; i < PL; ++i)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[i][k] = 0.0f;
  for (int rb = wi; rb < R; rb += 4 * WPE) {
    uint4 raw[4][PL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = rb + u * WPE, t = lo + rr;
      if (rr < R && t >= 0) load_row_raw<D>(token_row(p, b, sp, t, D), lane, raw[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = rb + u * WPE, t = lo + rr;
      if (rr >= R) break;
      if (t < 0) continue;
      const float a = expf(zbuf[e_local][rr] - zmax) * inv;
      float v[PL][8];
      unpack_row<D>(raw[u], lane, v);
#pragma unroll
      for (int i = 0; i < PL; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[i][k] = fmaf(a, v[i][k], acc[i][k]);
    }
  }

  if constexpr (WPE > 1) {
    // cross-warp sum in a fixed order (deterministic)
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      int c = lane + 32 * i;
      if (c < RowChunks<D>::kChunks)
#pragma unroll
        for (int k = 0; k < 8; ++k) red[warp][c * 8 + k] = acc[i][k];
    }
    __syncthreads();
    if (wi != 0) return;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      int c = lane + 32 * i;
      if (c < RowChunks<D>::kChunks)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float s = 0.0f;
          for (int wq = 0; wq < WPE; ++wq) s += red[e_local * WPE + wq][c * 8 + k];
          acc[i][k] = s;
        }
    }
  }

  const long long row = entry_row(p.paging, b, j, p.entries.num_rows);
  if (row < 0) {
    if (lane == 0) report(p.status, LCS_ERR_DEVICE_GUARD);
    return;
  }
  store_row<D>(p.entries, row, lane, acc);
}

// Score row of raw token t (per-channel weights): this call's score rows or the pending ring.
__device__ __forceinline__ const __nv_bfloat16* score_row(const CompressParams& p, int b, const SeqSpan& sp, int t,
                                                          int D) {
  if (t >= sp.n0()) return p.scores + (long long)(sp.q0 + t - sp.n0()) * D;
  return p.pending_scores + ((long long)b * p.pending_slots + (t % p.pending_slots)) * D;
}

// Compression for ratios up to 4 (CSA): a warp takes a run of kRollEntries consecutive entries of
// one sequence and streams their blocks of M rows through a three-slot ring of its own in shared
// memory (cp.async, 16 bytes per lane, each lane reading back only the pieces it copied), so that
// every raw row is read from memory once: block j-1 stays for entry j (overlapping windows) and
// block j+1 is in flight while entry j is formed.  The arithmetic of an entry is the same whichever
// warp or call forms it.  Scalar weights: z_t = (w . k_t as a warp sum) + bias[offset], the
// softmax over the rows that exist in row order, the weighted sum in row order.  Per-channel
// weights (PC): a slot also holds the block's score rows; per channel, z = score + bias[offset][c],
// the maximum over the rows, then the exponentials' sum and the exponential-weighted sum of the
// rows in row order, divided by that sum.
constexpr int kRollEntries = 16;
constexpr int kRollSlots = 3;

template <int D, int M, bool PC>
__global__ void __launch_bounds__(PC ? 128 : 256) compress_roll_kernel(CompressParams p) {
  constexpr int kWarps = PC ? 4 : 8;
  constexpr int PL = RowChunks<D>::kPerLane;
  constexpr int C = RowChunks<D>::kChunks;
  constexpr int kBlockBytes = (PC ? 2 : 1) * M * D * 2;
  extern __shared__ __align__(16) uint8_t roll_smem[];
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  const int j_first = sp.n0() / M, j_end = sp.n1 / M;
  const int ja = j_first + (blockIdx.x * kWarps + warp) * kRollEntries;
  const int jb = min(j_end, ja + kRollEntries);
  if (ja >= jb) return;
  const bool ov = p.overlap != 0;
  uint8_t* ring = roll_smem + warp * (kRollSlots * kBlockBytes);
  float wv[PL][8];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int c = lane + 32 * i;
#pragma unroll
    for (int k = 0; k < 8; ++k) wv[i][k] = (!PC && c < C) ? p.w[c * 8 + k] : 0.0f;
  }
  // block jj -> slot (jj + 1) % 3 (rows 0..M-1 the raw rows, M..2M-1 the score rows); this lane
  // copies its own chunks (a group per block, empty for blocks outside [0, jb))
  auto issue = [&](int jj) {
    if (jj >= 0 && jj < jb) {
      uint8_t* slot = ring + ((jj + 1) % kRollSlots) * kBlockBytes;
#pragma unroll
      for (int r = 0; r < (PC ? 2 * M : M); ++r) {
        const __nv_bfloat16* src = r < M ? token_row(p, b, sp, jj * M + r, D) : score_row(p, b, sp, jj * M + r - M, D);
#pragma unroll
        for (int i = 0; i < PL; ++i) {
          const int c = lane + 32 * i;
          if (c < C) cp_async16(slot + r * D * 2 + c * 16, src + c * 8);
        }
      }
    }
    cp_async_commit();
  };
  // row r of block jj (r >= M: its score rows) as fp32, this lane's chunks
  auto row_vals = [&](int jj, int r, float (&v)[PL][8]) {
    const uint8_t* slot = ring + ((jj + 1) % kRollSlots) * kBlockBytes;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int c = lane + 32 * i;
      const uint4 u = c < C ? *reinterpret_cast<const uint4*>(slot + r * D * 2 + c * 16) : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        v[i][2 * k] = f.x;
        v[i][2 * k + 1] = f.y;
      }
    }
  };
  auto block_z = [&](int jj, float (&z)[M]) {
#pragma unroll
    for (int r = 0; r < M; ++r) {
      float v[PL][8];
      row_vals(jj, r, v);
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < PL; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = fmaf(wv[i][k], v[i][k], acc);
      z[r] = warp_sum(acc);
    }
  };
  issue(ov ? ja - 1 : -1);
  issue(ja);
  issue(ja + 1);
  float zp[M], zc[M];
  if (!PC && ov && ja >= 1) {
    cp_async_wait<2>();
    block_z(ja - 1, zp);
  }
  for (int j = ja; j < jb; ++j) {
    cp_async_wait<1>();   // blocks j-1 and j have landed (block j+1 may still be in flight)
    constexpr int R2 = 2 * M;
    const bool prev = ov && j >= 1;   // rows of block j-1 exist and belong to the window
    float acc[PL][8];
#pragma unroll
    for (int i = 0; i < PL; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[i][k] = 0.0f;
    if constexpr (!PC) {
      block_z(j, zc);
      // softmax over the window rows that exist: block j-1 (offsets 0..M-1) then block j
      float z[R2];
      bool ex[R2];
#pragma unroll
      for (int r = 0; r < M; ++r) {
        ex[r] = prev;
        z[r] = ex[r] ? zp[r] + p.bias[r] : -INFINITY;
        ex[M + r] = true;
        z[M + r] = zc[r] + p.bias[ov ? M + r : r];
      }
      float zmax = -INFINITY;
#pragma unroll
      for (int r = 0; r < R2; ++r) zmax = fmaxf(zmax, z[r]);
      float zsum = 0.0f;
#pragma unroll
      for (int r = 0; r < R2; ++r) zsum += ex[r] ? expf(z[r] - zmax) : 0.0f;
      const float inv = 1.0f / zsum;
#pragma unroll
      for (int r = 0; r < R2; ++r) {
        if (!ex[r]) continue;
        const float a = expf(z[r] - zmax) * inv;
        float v[PL][8];
        row_vals(r < M ? j - 1 : j, r % M, v);
#pragma unroll
        for (int i = 0; i < PL; ++i)
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[i][k] = fmaf(a, v[i][k], acc[i][k]);
      }
#pragma unroll
      for (int r = 0; r < M; ++r) zp[r] = zc[r];
    } else {
      // per channel: z = score + bias[offset][channel] over the rows that exist
      float zmax[PL][8], zsum[PL][8];
#pragma unroll
      for (int i = 0; i < PL; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          zmax[i][k] = -INFINITY;
          zsum[i][k] = 0.0f;
        }
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
        for (int r = 0; r < R2; ++r) {
          if (r < M && !prev) continue;
          const int o = ov ? r : r - M;   // offset in the window (non-overlapping: block j only)
          if (o < 0) continue;
          float sv[PL][8];
          row_vals(r < M ? j - 1 : j, M + (r % M), sv);
          float v[PL][8];
          if (pass == 1) row_vals(r < M ? j - 1 : j, r % M, v);
#pragma unroll
          for (int i = 0; i < PL; ++i) {
            const int c = lane + 32 * i;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float z = sv[i][k] + (c < C ? p.bias[o * D + c * 8 + k] : 0.0f);
              if (pass == 0) {
                zmax[i][k] = fmaxf(zmax[i][k], z);
              } else {
                const float e = expf(z - zmax[i][k]);
                zsum[i][k] += e;
                acc[i][k] = fmaf(e, v[i][k], acc[i][k]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < PL; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[i][k] = zsum[i][k] > 0.0f ? acc[i][k] / zsum[i][k] : 0.0f;
    }
    const long long row = entry_row(p.paging, b, j, p.entries.num_rows);
    if (row < 0) {
      if (lane == 0) report(p.status, LCS_ERR_DEVICE_GUARD);
    } else {
      store_row<D>(p.entries, row, lane, acc);
    }
    issue(j + 2);   // into the slot of block j-1, whose last reader was entry j
  }
  cp_async_wait<0>();
}

// One warp per new token: keep it in the pending ring if a future entry needs it, and write
// its quantised row to new_rows (or to the window ring when new_rows is absent).
// grid: (ceil(max_new / 8), num_seqs), block 256.
template <int D>
__global__ void __launch_bounds__(256) compress_state_kernel(CompressParams p) {
  constexpr int PL = RowChunks<D>::kPerLane;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqSpan sp = seq_span(p.cu_new, p.seq_len, b);
  // without new_rows only the last state_tail tokens can matter (pending rows, window ring)
  const int first = (p.new_rows.nope == nullptr && p.state_tail > 0) ? max(0, sp.qn - p.state_tail) : 0;
  const int i = first + blockIdx.x * 8 + warp;
  if (i >= sp.qn) return;
  const int t = sp.n0() + i;
  const int m = p.m;
  const int full = sp.n1 / m;
  const int keep_lo = p.overlap ? (full - 1) * m : full * m;
  if (t < keep_lo && p.new_rows.nope == nullptr && t < sp.n1 - kWindow) return;   // neither kept nor stored
  const __nv_bfloat16* src = p.raw + (long long)(sp.q0 + i) * D;
  float v[PL][8];
  load_row<D>(src, lane, v);
  if (t >= keep_lo) {
    __nv_bfloat16* dst = p.pending_out + ((long long)b * p.pending_slots + (t % p.pending_slots)) * D;
#pragma unroll
    for (int k = 0; k < PL; ++k) {
      int c = lane + 32 * k;
      if (c < RowChunks<D>::kChunks)
        *reinterpret_cast<uint4*>(dst + c * 8) = *reinterpret_cast<const uint4*>(src + c * 8);
    }
    if (p.pending_scores != nullptr) {   // per-channel weights: the token's score row too
      const __nv_bfloat16* ssrc = p.scores + (long long)(sp.q0 + i) * D;
      __nv_bfloat16* sdst = p.pending_scores + ((long long)b * p.pending_slots + (t % p.pending_slots)) * D;
#pragma unroll
      for (int k = 0; k < PL; ++k) {
        int c = lane + 32 * k;
        if (c < RowChunks<D>::kChunks)
          *reinterpret_cast<uint4*>(sdst + c * 8) = *reinterpret_cast<const uint4*>(ssrc + c * 8);
      }
    }
  }
  if (p.new_rows.nope != nullptr) {
    long long r = (long long)sp.q0 + i;
    if (r >= p.new_rows.num_rows) {
      if (lane == 0) report(p.status, LCS_ERR_DEVICE_GUARD);
      return;
    }
    store_row<D>(p.new_rows, r, lane, v);
  } else if (t >= sp.n1 - kWindow) {
    long long r = (long long)b * kWindow + (t % kWindow);
    if (r >= p.window.num_rows) {
      if (lane == 0) report(p.status, LCS_ERR_DEVICE_GUARD);
      return;
    }
    store_row<D>(p.window, r, lane, v);
  }
}

// Copy this call's new rows into the window ring.  grid: (ceil(min(max_new,128)/8), num_seqs).
__global__ void __launch_bounds__(256) window_commit_kernel(const int32_t* cu_new, const int32_t* seq_len,
                                                           Rows src, Rows ring, int32_t* status) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqSpan sp = seq_span(cu_new, seq_len, b);
  const int ncopy = min(sp.qn, kWindow);
  const int i = blockIdx.x * 8 + warp;  // 0 .. ncopy-1, the last ncopy new tokens
  if (i >= ncopy) return;
  const int t = sp.n1 - ncopy + i;
  const long long s = (long long)sp.q0 + (t - sp.n0());
  const long long d = (long long)b * kWindow + (t % kWindow);
  if (s >= src.num_rows || d >= ring.num_rows) {
    if (lane == 0) report(status, LCS_ERR_DEVICE_GUARD);
    return;
  }
  const int D = src.dim;
  if (src.format == LCS_ROW_BF16) {
    const uint4* a = reinterpret_cast<const uint4*>(src.nope + s * D * 2);
    uint4* o = reinterpret_cast<uint4*>(ring.nope + d * D * 2);
    for (int c = lane; c < D / 8; c += 32) o[c] = a[c];
    return;
  }
  const uint4* a = reinterpret_cast<const uint4*>(src.nope + s * (D - kRope));
  uint4* o = reinterpret_cast<uint4*>(ring.nope + d * (D - kRope));
  for (int c = lane; c < (D - kRope) / 16; c += 32) o[c] = a[c];
  const uint4* ra = reinterpret_cast<const uint4*>(src.rope + s * kRope);
  uint4* ro = reinterpret_cast<uint4*>(ring.rope + d * kRope);
  if (lane < kRope / 8) ro[lane] = ra[lane];
  if (lane == 0) ring.scale[d] = src.scale[s];
}

// ----------------------------------------------------------------------------------------------
// launchers
// ----------------------------------------------------------------------------------------------

template <int D, int M, bool PC>
cudaError_t launch_roll(const CompressParams& p, int max_entries, cudaStream_t st) {
  constexpr int kWarps = PC ? 4 : 8;
  constexpr size_t smem = (size_t)kWarps * kRollSlots * (PC ? 2 : 1) * M * D * 2;
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(compress_roll_kernel<D, M, PC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid((max_entries + kWarps * kRollEntries - 1) / (kWarps * kRollEntries), p.num_seqs);
  compress_roll_kernel<D, M, PC><<<grid, kWarps * 32, smem, st>>>(p);
  return cudaGetLastError();
}

template <int D, bool PC>
cudaError_t launch_roll_m(const CompressParams& p, int max_entries, cudaStream_t st) {
  if (p.m == 4) return launch_roll<D, 4, PC>(p, max_entries, st);
  if (p.m == 2) return launch_roll<D, 2, PC>(p, max_entries, st);
  return launch_roll<D, 1, PC>(p, max_entries, st);
}

constexpr int kFewTokens = 16;

cudaError_t launch_compress(const CompressParams& p, int D, int max_new, cudaStream_t st) {
  const int R = p.overlap ? 2 * p.m : p.m;
  const int max_entries = max_new / p.m + 1;
  cudaError_t e;
  // the streaming kernel (a shared-memory ring per warp) for chunks and for per-channel weights;
  // a few new tokens per sequence (decode: at most one entry completes) with scalar weights take
  // a warp per entry and no shared memory, so that their CTAs fit on SMs next to the indexer's
  const bool pc = p.scores != nullptr;
  if ((p.m == 4 || p.m == 2 || p.m == 1) && (max_new > kFewTokens || pc)) {
    if (D == 512) e = pc ? launch_roll_m<512, true>(p, max_entries, st) : launch_roll_m<512, false>(p, max_entries, st);
    else e = pc ? launch_roll_m<128, true>(p, max_entries, st) : launch_roll_m<128, false>(p, max_entries, st);
  } else {
    const bool cta_per_entry = R > 16;
    const int epc = cta_per_entry ? 1 : 8;
    dim3 grid((max_entries + epc - 1) / epc, p.num_seqs);
    if (D == 512) {
      if (cta_per_entry) compress_entries_kernel<512, 8><<<grid, 256, 0, st>>>(p);
      else compress_entries_kernel<512, 1><<<grid, 256, 0, st>>>(p);
    } else {
      if (cta_per_entry) compress_entries_kernel<128, 8><<<grid, 256, 0, st>>>(p);
      else compress_entries_kernel<128, 1><<<grid, 256, 0, st>>>(p);
    }
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || max_new == 0) return e;
  // without new_rows only the last state_tail tokens of each sequence go to the pending ring or
  // the window ring: launch warps for those alone
  const int warps = (p.new_rows.nope == nullptr && p.state_tail > 0 && p.state_tail < max_new) ? p.state_tail : max_new;
  dim3 g2((warps + 7) / 8, p.num_seqs);
  if (D == 512) compress_state_kernel<512><<<g2, 256, 0, st>>>(p);
  else compress_state_kernel<128><<<g2, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_window_commit(const int32_t* cu_new, const int32_t* seq_len, int num_seqs, int max_new,
                                 const Rows& src, const Rows& ring, int32_t* status, cudaStream_t st) {
  int n = max_new < kWindow ? max_new : kWindow;
  if (n <= 0) return cudaSuccess;
  dim3 grid((n + 7) / 8, num_seqs);
  window_commit_kernel<<<grid, 256, 0, st>>>(cu_new, seq_len, src, ring, status);
  return cudaGetLastError();
}

}  // namespace lcsa
