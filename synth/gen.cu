// On-device implementation of the seeded generator defined in synth/__init__.py (SplitMix64
// output function, Irwin-Hall bf16 normals, uniform E2M1 codes, UE8M0 scales).  Used to fill
// large synthetic inputs directly in HBM; it holds no step of the attention method.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t start, uint64_t n, __nv_bfloat16* out) {
  const float scale = __uint_as_float(0x37DDB3D7u);
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t u = draw(key, start + i);
    const int s = (int)(u & 0xFFFF) + (int)((u >> 16) & 0xFFFF) + (int)((u >> 32) & 0xFFFF) + (int)(u >> 48) - 131070;
    out[i] = __float2bfloat16_rn(__fmul_rn((float)s, scale));
  }
}

__constant__ uint8_t kCodes[15] = {0, 1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15};

// codes start .. start+2n-1 packed two per byte (even code in the low nibble)
__global__ void e2m1_packed_kernel(uint64_t key, uint64_t start, uint64_t n_bytes, uint8_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n_bytes; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint8_t lo = kCodes[draw(key, start + 2 * i) % 15];
    const uint8_t hi = kCodes[draw(key, start + 2 * i + 1) % 15];
    out[i] = (uint8_t)(lo | (hi << 4));
  }
}

__global__ void ue8m0_kernel(uint64_t key, uint64_t start, uint64_t n, int lo, int span, uint8_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)(127 + lo + (int)(draw(key, start + i) % (uint64_t)span));
}

uint64_t stream_key(uint32_t seed, uint32_t tid) {
  uint64_t z = ((uint64_t)seed << 32) | tid;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

unsigned grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  return (unsigned)(g > 65536 ? 65536 : (g == 0 ? 1 : g));
}

}  // namespace

extern "C" {

int synth_normal_bf16(uint32_t seed, uint32_t tid, uint64_t start, uint64_t n, void* out, void* stream) {
  if (n == 0) return 0;
  normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(stream_key(seed, tid), start, n,
                                                                     (__nv_bfloat16*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

int synth_e2m1_packed(uint32_t seed, uint32_t tid, uint64_t start_code, uint64_t n_bytes, void* out, void* stream) {
  if (n_bytes == 0) return 0;
  e2m1_packed_kernel<<<grid_for(n_bytes), 256, 0, (cudaStream_t)stream>>>(stream_key(seed, tid), start_code, n_bytes,
                                                                          (uint8_t*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

int synth_ue8m0(uint32_t seed, uint32_t tid, uint64_t start, uint64_t n, int lo, int hi, void* out, void* stream) {
  if (n == 0) return 0;
  ue8m0_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(stream_key(seed, tid), start, n, lo, hi - lo + 1,
                                                              (uint8_t*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

}  // extern "C"
