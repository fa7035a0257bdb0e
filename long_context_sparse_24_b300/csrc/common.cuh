// Device helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "lcsa.h"

namespace lcsa {

constexpr int kWindow = LCSA_WINDOW;
constexpr int kRope = LCSA_ROPE_DIMS;
constexpr int kBlockTokens = LCSA_BLOCK_TOKENS;

// First device-side error wins; the caller reads the word after the stream completes.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Span of sequence b in the batch: first global token index, new-token count, length after.
struct SeqSpan {
  int q0;   // cu_new[b]
  int qn;   // new tokens of the sequence
  int n1;   // seq_len[b]
  __device__ __forceinline__ int n0() const { return n1 - qn; }
};

__device__ __forceinline__ SeqSpan seq_span(const int32_t* cu_new, const int32_t* seq_len, int b) {
  SeqSpan s;
  s.q0 = cu_new[b];
  s.qn = cu_new[b + 1] - s.q0;
  s.n1 = seq_len[b];
  return s;
}

// Sequence of global query q (cu_new non-decreasing), found by the whole CTA: cu_new is staged in
// shared memory with one parallel load when the batch has at most `cap` sequences (a binary search
// over global memory costs a dependent load per step), else searched in global memory.  Every
// thread of the CTA calls it; scratch: cap + 1 ints of shared memory, free again on return.
__device__ __forceinline__ int find_seq_block(const int32_t* cu_new, int num_seqs, int q, int* scratch, int cap) {
  int lo = 0, hi = num_seqs - 1;
  if (num_seqs + 1 <= cap) {
    for (int i = threadIdx.x; i <= num_seqs; i += blockDim.x) scratch[i] = cu_new[i];
    __syncthreads();
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (scratch[mid] <= q) lo = mid; else hi = mid - 1;
    }
    __syncthreads();
    return lo;
  }
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_new[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The sequence b of global query q and its span, found by the whole CTA with cu_new and seq_len
// staged in shared memory by one parallel load (scratch: 2 * num_seqs + 1 ints when that is at
// most `cap`; otherwise read from global memory).
__device__ __forceinline__ SeqSpan find_seq_span(const int32_t* cu_new, const int32_t* seq_len, int num_seqs, int q,
                                                 int* scratch, int cap, int* b_out) {
  if (2 * num_seqs + 1 > cap) {
    const int b = find_seq_block(cu_new, num_seqs, q, scratch, 0);
    *b_out = b;
    return seq_span(cu_new, seq_len, b);
  }
  for (int i = threadIdx.x; i <= num_seqs; i += blockDim.x) scratch[i] = cu_new[i];
  for (int i = threadIdx.x; i < num_seqs; i += blockDim.x) scratch[num_seqs + 1 + i] = seq_len[i];
  __syncthreads();
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (scratch[mid] <= q) lo = mid; else hi = mid - 1;
  }
  SeqSpan s;
  s.q0 = scratch[lo];
  s.qn = scratch[lo + 1] - s.q0;
  s.n1 = scratch[num_seqs + 1 + lo];
  __syncthreads();
  *b_out = lo;
  return s;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The end of a softmax over rows with a per-head sink logit folded in (one more term e^sink in the
// denominator that carries no value; sink in natural-log units, NULL = none).  The rows give their
// running max m and sum l of 2^(logit - m) (logits in base 2); f turns the rows' weighted sum
// (relative to m) into the output and lse2 is the log-sum-exp in base 2.  Without a sink f = 1/l.
struct SoftmaxNorm {
  float f;
  float lse2;
};
__device__ __forceinline__ SoftmaxNorm softmax_norm(float m, float l, const float* sink, int h) {
  if (sink == nullptr) return SoftmaxNorm{l > 0.0f ? 1.0f / l : 0.0f, l > 0.0f ? m + log2f(l) : -INFINITY};
  const float s2 = sink[h] * 1.4426950408889634f;
  const float mx = l > 0.0f ? fmaxf(m, s2) : s2;
  const float a = l > 0.0f ? exp2f(m - mx) : 0.0f;
  const float lp = fmaf(l, a, exp2f(s2 - mx));
  return SoftmaxNorm{a / lp, mx + log2f(lp)};
}

// Programmatic dependent launch (PTX griddepcontrol).  A kernel launched as a programmatic
// dependent of the preceding kernel in its stream may start before that kernel ends: it must not
// read what that kernel writes before grid_dependency_wait(), which returns once the preceding
// grid has completed and its writes are visible (at once for a kernel launched normally).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the dependent grid start once every CTA of this grid has issued this or exited.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Row set view (mirrors lcs_rows).
struct Rows {
  int format;
  int dim;
  long long num_rows;
  uint8_t* nope;
  __nv_bfloat16* rope;
  float* scale;
};

__host__ __device__ inline Rows make_rows(const lcs_rows& r) {
  Rows v;
  v.format = r.format;
  v.dim = r.dim;
  v.num_rows = r.num_rows;
  v.nope = static_cast<uint8_t*>(r.nope);
  v.rope = static_cast<__nv_bfloat16*>(r.rope);
  v.scale = r.scale;
  return v;
}

struct Paging {
  int epb;                 // entries per block
  int max_blocks;          // per sequence
  const int32_t* table;
};

__host__ __device__ inline Paging make_paging(const lcs_paging& p) {
  Paging v;
  v.epb = p.entries_per_block;
  v.max_blocks = p.max_blocks_per_seq;
  v.table = p.block_table;
  return v;
}

// Physical row of entry j of sequence b, or -1 when unmapped / out of range.
__device__ __forceinline__ long long entry_row(const Paging& pg, int b, int j, long long num_rows) {
  int blk = j / pg.epb;
  if (blk >= pg.max_blocks) return -1;
  int phys = pg.table[(long long)b * pg.max_blocks + blk];
  if (phys < 0) return -1;
  long long row = (long long)phys * pg.epb + (j - blk * pg.epb);
  return row < num_rows ? row : -1;
}

// ---------------------------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------------------------

// The attention kernels multiply probabilities by a row's FP8 scale s_r and by 2^8 in f16
// (p * s_r * 2^8 <= 65504 needs s_r < 256), and the tensor-core kernels divide the RoPE dims by
// s_r in f16 (|rope| / s_r <= 65504).  Rows outside these ranges are left out of the softmax and
// reported as LCS_ERR_DEVICE_GUARD.
constexpr float kMaxRowScale = 256.0f;

// True when one of the f16 values is infinite or NaN (exponent bits all set).
__device__ __forceinline__ bool f16x2_nonfinite(uint32_t w) {
  return (w & 0x7C00u) == 0x7C00u || (w & 0x7C000000u) == 0x7C000000u;
}
__device__ __forceinline__ bool f16x8_nonfinite(uint4 v) {
  return f16x2_nonfinite(v.x) || f16x2_nonfinite(v.y) || f16x2_nonfinite(v.z) || f16x2_nonfinite(v.w);
}

// fp32 pair -> two E4M3 codes (round to nearest even, saturate to +-448), packed low = a.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  // cvt packs its first source operand into the upper byte.
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Two E4M3 codes (low byte first) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

__device__ __forceinline__ float ue8m0_to_f32(uint32_t e) {
  // 2^(e-127); e = 0 is the subnormal 2^-127; 255 (NaN in the MX formats) is not produced here.
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// Order-preserving map of an fp32 score onto uint32 (larger score -> larger key).
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s == 0.0f ? 0.0f : s);  // -0 and +0 share one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// ---------------------------------------------------------------------------------------------
// Warp-level MMA and shared-memory matrix loads (legacy warp MMA; tcgen05 kernels live apart)
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A(16x32 e4m3, row) * B(32x8 e4m3, col), fp32, C = 0.
__device__ __forceinline__ void mma_e4m3_zero(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// cp.async 16 / 4 bytes global -> shared (L2-only for 16-byte copies).  The memory clobbers keep
// the compiler from moving shared-memory reads across a copy's issue or its wait.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace lcsa
