// Block-scaled FP4 quantisation of BF16 rows: the production of the lightning indexer's keys and
// queries.
//
// Defined by: m.x-techcon.com/article/133366, section 4 "FP4量化感知训练" (the indexer's QK path
// runs in FP4) and the latetalk.qiaomu.ai notes on V4's attention (block-wise scales); the values
// of E2M1 from chenxutan.com/d/4230, section 6.2.  The pages fix the format -- E2M1 codes with one
// power-of-two (UE8M0) scale per 32 elements -- but not how the scale is chosen.  Here: the
// smallest power of two 2^e with amax <= 6 * 2^e (no element saturates), e clamped to the UE8M0
// range [-127, 127] (all-zero blocks: e = -127); each element is x / 2^e rounded to the nearest
// E2M1 value, ties to the code with mantissa bit 0; zero is stored as +0.
//
// A thread per 16 elements (two 16-byte loads, one 8-byte store of codes), two threads per
// 32-element block sharing its amax through one shuffle.
#include "kernels.cuh"

namespace lcsa {

namespace {

constexpr int kQuantThreads = 256;

// E2M1 magnitude code (0..7) of |v| <= 6, round to nearest, ties to the even code: the number of
// midpoints between neighbouring values 0, 0.5, 1, 1.5, 2, 3, 4, 6 that lie below a, where a
// value at a midpoint goes to the even code (0, 2, 4, 6) -- branch-free.
__device__ __forceinline__ uint32_t e2m1_code_rne(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
         (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
}

__global__ void __launch_bounds__(kQuantThreads) quantize_e2m1_kernel(const uint4* __restrict__ x, long long n16,
                                                                      uint2* __restrict__ codes,
                                                                      uint8_t* __restrict__ scales) {
  // thread t: elements 16t .. 16t+15 of the flattened rows (two 16-byte loads, one 8-byte store
  // of codes); two consecutive threads hold one 32-element block (rows are whole blocks)
  const long long t = (long long)blockIdx.x * kQuantThreads + threadIdx.x;
  const bool valid = t < n16;
  const uint4 r0 = valid ? x[2 * t] : make_uint4(0u, 0u, 0u, 0u);
  const uint4 r1 = valid ? x[2 * t + 1] : make_uint4(0u, 0u, 0u, 0u);
  float v[16];
  const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  // smallest e with 6 * 2^e >= amax: amax = m * 2^k, m in [1, 2): e = k - 2 when m <= 1.5, else
  // k - 1; zero and subnormal amax (below 6 * 2^-127 either way) take the clamp -127
  const uint32_t bits = __float_as_uint(amax);
  const int expb = (int)(bits >> 23);
  int e = -127;
  if (expb > 0) e = (expb - 127) - 2 + ((bits & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  e = max(-127, min(127, e));
  // 2^-e (normal for e <= 126, the subnormal 2^-127 for e = 127); |v| * 2^-e is exact wherever
  // the result can round to a non-zero code (below 2^-126 it rounds to 0)
  const float inv = e < 127 ? __uint_as_float((uint32_t)(127 - e) << 23) : __uint_as_float(0x00400000u);
  uint32_t lo = 0u, hi = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint32_t c = e2m1_code_rne(fabsf(v[i]) * inv);
    if (c != 0u && v[i] < 0.0f) c |= 8u;
    if (i < 8) lo |= c << (4 * i);                // even element in the low nibble of its byte
    else hi |= c << (4 * (i - 8));
  }
  if (valid) {
    codes[t] = make_uint2(lo, hi);
    if ((t & 1) == 0) scales[t >> 1] = (uint8_t)(e + 127);
  }
}

}  // namespace

}  // namespace lcsa

extern "C" lcs_status lcs_quantize_e2m1(const void* x, int64_t rows, int32_t r, uint8_t* codes, uint8_t* scales,
                                        void* stream) {
  using namespace lcsa;
  if (rows < 0 || r <= 0 || (r & 31) != 0 || r > 4096) return LCS_ERR_UNSUPPORTED;
  if (rows == 0) return LCS_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return LCS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return LCS_ERR_ALIGNMENT;
  const long long n16 = rows * (r >> 4);
  const long long ctas = (n16 + kQuantThreads - 1) / kQuantThreads;
  if (ctas > 0x7fffffffll) return LCS_ERR_UNSUPPORTED;
  quantize_e2m1_kernel<<<(unsigned)ctas, kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(x), n16, reinterpret_cast<uint2*>(codes), scales);
  return cudaGetLastError() == cudaSuccess ? LCS_OK : LCS_ERR_CUDA;
}

// ----------------------------------------------------------------------------------------------
// Attention sink: a per-head logit that joins every softmax denominator and carries no value
// (the csdn attention-details table names an attention sink without defining it; this is the
// common learned-sink definition).  Applied after the attention call from its outputs and their
// log-sum-exp: o' = o / (1 + exp(sink_h - lse)), lse' = log(exp(lse) + exp(sink_h)).
// ----------------------------------------------------------------------------------------------

namespace lcsa {
namespace {

constexpr int kSinkWarps = 4;

__global__ void __launch_bounds__(kSinkWarps * 32) attention_sink_kernel(__nv_bfloat16* __restrict__ out,
                                                                         float* __restrict__ lse,
                                                                         const float* __restrict__ sink,
                                                                         long long pairs, int heads, int dim) {
  const long long pr = (long long)blockIdx.x * kSinkWarps + (threadIdx.x >> 5);   // (query, head)
  if (pr >= pairs) return;                                                      // warp-uniform
  const int lane = threadIdx.x & 31;
  const int h = (int)(pr % heads);
  const float l = lse[pr], s = sink[h];
  const float d = s - l;
  // 1 / (1 + e^d) without overflow, and log(e^l + e^s) = max + log1p(e^-|l - s|)
  const float f = d > 0.0f ? expf(-d) / (1.0f + expf(-d)) : 1.0f / (1.0f + expf(d));
  uint4* row = reinterpret_cast<uint4*>(out + pr * dim);
  for (int i = lane; i < dim / 8; i += 32) {
    uint4 v = row[i];
    uint32_t* w = &v.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
      const __nv_bfloat162 b = __floats2bfloat162_rn(a.x * f, a.y * f);
      w[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    row[i] = v;
  }
  if (lane == 0) lse[pr] = fmaxf(l, s) + log1pf(expf(-fabsf(l - s)));
}

}  // namespace
}  // namespace lcsa

extern "C" lcs_status lcs_attention_sink(void* out, float* out_lse, const float* sink, int64_t total_new,
                                         int32_t heads, int32_t dim, void* stream) {
  using namespace lcsa;
  if (total_new < 0 || heads <= 0 || dim <= 0 || (dim & 7) != 0) return LCS_ERR_UNSUPPORTED;
  if (total_new == 0) return LCS_OK;
  if (out == nullptr || out_lse == nullptr || sink == nullptr) return LCS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 15u) return LCS_ERR_ALIGNMENT;
  const long long pairs = total_new * (long long)heads;
  const long long ctas = (pairs + kSinkWarps - 1) / kSinkWarps;
  if (ctas > 0x7fffffffll) return LCS_ERR_UNSUPPORTED;
  attention_sink_kernel<<<(unsigned)ctas, kSinkWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<__nv_bfloat16*>(out), out_lse, sink, pairs, heads, dim);
  return cudaGetLastError() == cudaSuccess ? LCS_OK : LCS_ERR_CUDA;
}
