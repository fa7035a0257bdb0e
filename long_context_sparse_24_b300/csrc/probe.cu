// Tensor-pipe throughput probe: the denominators of the indexer's and the attention's tensor
// roofline, measured with the same tcgen05 instruction forms the library's kernels issue.
//
// Not a step of the method.  Every CTA (one per SM) keeps one 128-row A tile and one N = 256 row
// B tile in shared memory and issues back-to-back MMAs of M = 128, N = 256 into two tensor-memory
// accumulators, committing each group of 64 to a barrier before reusing its accumulator:
//   kind 0: kind::f8f6f4 with E2M1 operands in the "16 x U4 in 16 bytes" K-major form (the
//           indexer scorers' MMA), K = 32 per instruction;
//   kind 1: kind::f16 with F16 operands (the attention kernels' MMA), K = 16 per instruction;
//   kind 2: kind::mxf4, block-scaled E2M1 operands packed two codes a byte (64-byte swizzle), a
//           UE8M0 scale per 32 codes from tensor memory (all 2^0 here), K = 64 per instruction,
//           N = 240 (two accumulators and the scale factors share the 512 tensor-memory columns).
// The caller times the launch (CUDA events) and divides 2 * 128 * N * K * mmas * CTAs by it.
// Operand values are zeros; waits are bounded like every wait of the library.
#include "kernels.cuh"
#include "sm100.cuh"

namespace lcsa {

namespace {

constexpr int kProbeN = 256;
constexpr int kProbeNmx = 240;    // kind 2: N, and the accumulators' columns
constexpr int kProbeGroup = 64;   // MMAs per commit

__global__ void __launch_bounds__(128, 1) mma_probe_kernel(int kind, int mmas, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  constexpr int kA = 0;                       // 128 rows x 128 B
  constexpr int kB = 128 * 128;               // 256 rows x 128 B
  constexpr int kBar = kB + kProbeN * 128;    // u64 x 2
  constexpr int kMisc = kBar + 16;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < (kBar / 16); i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(sbase + kBar, 1);
    mbar_init(sbase + kBar + 8, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(sbase + kMisc, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kMisc);
  // kind 2: scale factors 2^0 (UE8M0 127) in columns 480..487 of every lane
  const uint32_t tm_sf = tmem + 2 * kProbeNmx;
  if (kind == 2) {
    tmem_st4_fill(tm_sf + ((uint32_t)(warp * 32) << 16), 0x7F7F7F7Fu);
    tmem_st4_fill(tm_sf + 4 + ((uint32_t)(warp * 32) << 16), 0x7F7F7F7Fu);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (tid == 0) {
    const uint64_t ad = smem_desc_sw128(sbase + kA), bd = smem_desc_sw128(sbase + kB);
    const uint32_t id8 = idesc_f8f6f4(5, 5, 128, kProbeN);
    const uint32_t id16 = idesc_f16(0, 128, kProbeN);
    const uint32_t idmx = idesc_mxf4(128, kProbeNmx);
    const uint64_t ad64 = smem_desc_sw64(sbase + kA), bd64 = smem_desc_sw64(sbase + kB);
    const int groups = (mmas + kProbeGroup - 1) / kProbeGroup;
    bool ok = true;
    int issued = 0;
    for (int g = 0; g < groups && ok; ++g) {
      const int acc = g & 1;
      // the accumulator's previous group has completed before it is overwritten
      if (g >= 2) ok = mbar_wait(sbase + kBar + 8 * acc, ((g >> 1) - 1) & 1, status);
      if (!ok) break;
      tc_fence_after_sync();
      for (int i = 0; i < kProbeGroup; ++i) {
        const uint32_t step = (uint32_t)(i & 3);   // four K steps cover the 128-byte rows
        if (kind == 0)
          tc_mma_f8f6f4(tmem + acc * kProbeN, ad + 2 * step, bd + 2 * step, id8, i > 0 ? 1u : 0u);
        else if (kind == 1)
          tc_mma_f16(tmem + acc * kProbeN, ad + 2 * step, bd + 2 * step, id16, i > 0 ? 1u : 0u);
        else   // two K steps of 32 bytes cover the 64-byte rows
          tc_mma_mxf4(tmem + acc * kProbeNmx, ad64 + 2 * (step & 1), bd64 + 2 * (step & 1), idmx, tm_sf, tm_sf + 4,
                      i > 0 ? 1u : 0u);
      }
      tc_commit(sbase + kBar + 8 * acc);
      ++issued;
    }
    // every group issued has completed before tensor memory is released
    for (int a = 0; a < 2 && issued > a; ++a) {
      const int last = ((issued - 1 - a) >> 1) << 1 | a;   // the last group on accumulator a
      mbar_wait(sbase + kBar + 8 * a, (last >> 1) & 1, status);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

}  // namespace lcsa

extern "C" lcs_status lcs_mma_probe(int32_t kind, int32_t mmas_per_cta, int32_t ctas, int32_t* dev_status,
                                    void* stream) {
  using namespace lcsa;
  if (kind < 0 || kind > 2 || mmas_per_cta < kProbeGroup || ctas < 1 || ctas > 65535) return LCS_ERR_UNSUPPORTED;
  // more shared memory than two CTAs of an SM could share: one CTA per SM, so that no CTA waits
  // in its tensor-memory allocation for another
  constexpr size_t smem = 120 * 1024;
  static_assert(smem >= 128 * 128 + kProbeN * 128 + 32 + 1024, "operands");
  static PerDeviceOnce attr;
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return LCS_ERR_CUDA;
  mma_probe_kernel<<<ctas, 128, smem, static_cast<cudaStream_t>(stream)>>>(kind, mmas_per_cta, dev_status);
  return cudaGetLastError() == cudaSuccess ? LCS_OK : LCS_ERR_CUDA;
}
