// csa_index_topk_noalloc: the indexer top-k for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to allocate: code that runs while another
// framework is capturing a CUDA graph (cudaMalloc is illegal during capture), serving runtimes
// that hand out all device memory once at start-up from their own pool and forbid later
// allocations, and plugin hosts that give a plugin only the tensors of the current call.
// Such a caller cannot provide the workspace that csa_index_topk needs.  This entry point uses
// a fixed scratch array that lives in the library's own device image instead: it is created
// when the library's module is loaded on a GPU and stays reserved on every GPU that loads the
// library until the process exits.
//
// The array's name in host code is only a host-side stand-in, not a device address, so the
// device address is looked up with cudaGetSymbolAddress, once per device, with that device
// current, and then cached.  The first call on a device does that lookup; make that first
// call before any stream capture starts.
//
// All calls share the one array, which keeps whatever the previous call left in it.  Its leading
// per-sequence counters and per-query thresholds must be zero when a call starts: the array is zero when the library's
// module is loaded, and every call that completes leaves them at zero again (on the path that
// writes every score instead, the histograms are cleared by a memset of this array, which is not
// an allocation).  A call with LCS_INDEX_SELECT_ONLY reads what the last LCS_INDEX_SCORE_ONLY call
// left in the array.  Two calls whose kernels overlap on the GPU (different streams, or different
// host threads on the same device without ordering) race on the array and give wrong results:
// order them.
#include <mutex>

#include "kernels.cuh"

namespace {

__device__ __align__(256) uint8_t g_index_scratch[LCSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
lcs_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LCS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || p == nullptr) return LCS_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LCS_OK;
}

}  // namespace

extern "C" lcs_status csa_index_topk_noalloc(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale,
                                             const float* head_w, int32_t heads, const lcs_index_keys* keys,
                                             const lcs_paging* paging, int32_t m, int32_t k, int32_t flags,
                                             int32_t* out_idx, int32_t* out_cnt, int32_t* dev_status,
                                             void* stream) {
  if (batch == nullptr || keys == nullptr || paging == nullptr) return LCS_ERR_INVALID_ARG;
  if (m <= 0 || k < 1) return LCS_ERR_UNSUPPORTED;
  if (lcs_index_topk_workspace(batch, heads, keys, paging, m, k) > (size_t)LCSA_NOALLOC_SCRATCH_BYTES)
    return LCS_ERR_WORKSPACE;
  void* scratch = nullptr;
  lcs_status s = scratch_on_current_device(&scratch);
  if (s != LCS_OK) return s;
  return csa_index_topk(batch, q_fp4, q_scale, head_w, heads, keys, paging, m, k, flags, out_idx, out_cnt, scratch,
                        (size_t)LCSA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
