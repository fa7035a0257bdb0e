// Staging copies between device-accessible buffers with the SMs' own loads and stores.
//
// Not a step of the method: the input side of a serving step.  A step's inputs usually arrive in
// pinned host memory; the copy engine moves a few MB from there at a fraction of the link's rate
// (measured on B300: about 12 GB/s for 2 MB host-to-device, against about 43 GB/s for the same
// bytes read by a kernel from the mapped pinned pages), so a step's host inputs are gathered by
// one kernel that reads the pinned pages directly, up to kMaxCopies buffers per launch.  (Pages
// the CPU has just written are read several times slower by either route; the kernel stays about
// twice as fast as the copy engine there.)
#include <cstring>

#include "kernels.cuh"

namespace lcsa {

namespace {

constexpr int kMaxCopies = 8;

struct CopyList {
  const uint8_t* src[kMaxCopies];
  uint8_t* dst[kMaxCopies];
  unsigned long long bytes[kMaxCopies];
  int n;
};

// grid: (CTAs per copy, copies).  16-byte pieces when both ends are 16-byte aligned, bytes otherwise.
__global__ void __launch_bounds__(256) stage_copy_kernel(const __grid_constant__ CopyList c) {
  const int i = blockIdx.y;
  const uint8_t* src = c.src[i];
  uint8_t* dst = c.dst[i];
  const unsigned long long n = c.bytes[i];
  const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0) {
    const unsigned long long n16 = n >> 4;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    // four pieces a thread loaded before any is stored: their reads (host memory over the link,
    // for pinned sources) are in flight together
    for (unsigned long long k0 = tid; k0 < n16; k0 += 4 * stride) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (k0 + u * stride < n16) v[u] = s4[k0 + u * stride];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (k0 + u * stride < n16) d4[k0 + u * stride] = v[u];
    }
    for (unsigned long long k = (n16 << 4) + tid; k < n; k += stride) dst[k] = src[k];
  } else {
    for (unsigned long long k = tid; k < n; k += stride) dst[k] = src[k];
  }
}

// The device address of a buffer: pinned host memory maps to its device alias, device memory
// (and managed memory) is used as is; NULL when the device cannot reach it.
const void* device_alias(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) {
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return d;
  }
  return nullptr;
}

}  // namespace

}  // namespace lcsa

extern "C" lcs_status lcs_stage_copy(int32_t n, void* const* dst, const void* const* src, const size_t* bytes,
                                     void* stream) {
  using namespace lcsa;
  if (n < 0 || n > kMaxCopies) return LCS_ERR_UNSUPPORTED;
  if (n == 0) return LCS_OK;
  if (dst == nullptr || src == nullptr || bytes == nullptr) return LCS_ERR_INVALID_ARG;
  CopyList c;
  std::memset(&c, 0, sizeof(c));
  unsigned long long most = 0;
  for (int i = 0; i < n; ++i) {
    if (bytes[i] == 0) {
      c.src[i] = nullptr;
      c.dst[i] = nullptr;
      continue;
    }
    if (dst[i] == nullptr || src[i] == nullptr) return LCS_ERR_INVALID_ARG;
    const void* s = device_alias(src[i]);
    const void* d = device_alias(dst[i]);
    if (s == nullptr || d == nullptr) return LCS_ERR_INVALID_ARG;
    c.src[i] = static_cast<const uint8_t*>(s);
    c.dst[i] = static_cast<uint8_t*>(const_cast<void*>(d));
    c.bytes[i] = bytes[i];
    if (bytes[i] > most) most = bytes[i];
  }
  c.n = n;
  if (most == 0) return LCS_OK;
  // enough 16-byte pieces in flight to cover the link's latency: one CTA per 16 KB, capped
  unsigned long long ctas = (most + 16383) / 16384;
  if (ctas > 1184) ctas = 1184;
  stage_copy_kernel<<<dim3((unsigned)ctas, n), 256, 0, static_cast<cudaStream_t>(stream)>>>(c);
  return cudaGetLastError() == cudaSuccess ? LCS_OK : LCS_ERR_CUDA;
}

