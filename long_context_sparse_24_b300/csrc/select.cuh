// Block-level exact selection of the k largest 64-bit keys, for the indexer's top-k.
//
// A candidate is key64 = (order-preserving score key << 32) | ~j, so that larger scores come
// first and, among equal scores, lower entry indices j (x-techcon section 2, CSA step 2: each
// query keeps the k highest-scoring entries; ties go to the lower index).  Keys are unique, so
// "the k largest keys" is one exact set.
//
// The helpers run on a group of NT threads: the whole CTA (ID 0, __syncthreads) or the first NT
// threads (a named barrier ID > 0).  Every thread of the group calls every helper.
#pragma once

#include "common.cuh"

namespace lcsa {

template <int NT, int ID>
__device__ __forceinline__ void group_sync() {
  if constexpr (ID == 0) {
    __syncthreads();
  } else {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(NT) : "memory");
  }
}

// Inclusive prefix sum of one int per thread over the group; *total gets the group's sum.
// warp_tot: NT/32 ints of shared memory.
template <int NT, int ID>
__device__ __forceinline__ int group_scan_incl(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  group_sync<NT, ID>();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const int t = warp_tot[w];
    before += w < warp ? t : 0;
    all += t;
  }
  group_sync<NT, ID>();
  *total = all;
  return before + x;
}

// Shared scratch of the selection helpers.
template <int NT>
struct SelScratch {
  uint32_t hist[256];
  int warp_tot[NT / 32];
  int found[3];      // digit, keys above it, keys in it
  int count;         // append counter
  unsigned long long span[2 * (NT / 32)];   // per-warp max / min of the keys
};

// Adds one to hist[bin] for every lane that passes `take`, one shared atomic per distinct bin of
// the warp (keys of a selection often share their leading digits: per-lane atomics on one address
// would serialise).  The whole warp must call.
__device__ __forceinline__ void warp_hist_add(bool take, uint32_t bin, uint32_t* hist) {
  const unsigned act = __ballot_sync(0xffffffffu, take);
  if (!take) return;
  const unsigned same = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == (unsigned)(__ffs(same) - 1)) atomicAdd(&hist[bin], (uint32_t)__popc(same));
}

// Key sources for the selection: groups of keys, count(g) keys in group g.
struct SmemKeys {            // one array
  const uint64_t* buf;
  int n;
  __device__ __forceinline__ int groups() const { return 1; }
  __device__ __forceinline__ int count(int) const { return n; }
  __device__ __forceinline__ uint64_t key(int, int i) const { return buf[i]; }
};
struct RunLists {            // lists of up to `stride` keys each, counts in shared memory
  const uint64_t* keys;      // global, written by other CTAs of the grid: read through L2
  const int* cnt;
  int lists;
  int stride;
  __device__ __forceinline__ int groups() const { return lists; }
  __device__ __forceinline__ int count(int g) const { return cnt[g]; }
  __device__ __forceinline__ uint64_t key(int g, int i) const {
    return __ldcg(reinterpret_cast<const unsigned long long*>(keys) + (long long)g * stride + i);
  }
};

// The threshold tau with exactly k of the source's keys >= tau (k <= number of keys; keys
// unique).  Most-significant-digit radix selection, 8 bits per pass, stopping as soon as the digit
// bin that holds the k-th key is taken whole (with unique keys that happens at the last digit at
// the latest).
template <int NT, int ID, typename Src>
__device__ uint64_t kth_largest_key(int k, const Src& src, SelScratch<NT>& sc) {
  static_assert(NT >= 256, "one bin per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the leading bits all keys share need no pass: start at the byte of the highest bit in which
  // the largest and the smallest key differ
  unsigned long long kmax = 0ull, kmin = ~0ull;
  for (int g = 0; g < src.groups(); ++g) {
    const int n = src.count(g);
    for (int i = tid; i < n; i += NT) {
      const unsigned long long u = src.key(g, i);
      kmax = u > kmax ? u : kmax;
      kmin = u < kmin ? u : kmin;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long a = __shfl_xor_sync(0xffffffffu, kmax, o), b = __shfl_xor_sync(0xffffffffu, kmin, o);
    kmax = a > kmax ? a : kmax;
    kmin = b < kmin ? b : kmin;
  }
  if (lane == 0) {
    sc.span[2 * warp] = kmax;
    sc.span[2 * warp + 1] = kmin;
  }
  group_sync<NT, ID>();
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    kmax = sc.span[2 * w] > kmax ? sc.span[2 * w] : kmax;
    kmin = sc.span[2 * w + 1] < kmin ? sc.span[2 * w + 1] : kmin;
  }
  if (kmax == kmin) return kmax;   // one key (k == 1)
  int shift = (63 - __clzll((long long)(kmax ^ kmin))) & ~7;
  uint64_t prefix = shift >= 56 ? 0ull : (kmax & (~0ull << (shift + 8)));
  int remaining = k;
  for (;; shift -= 8) {
    const uint64_t hi = shift >= 56 ? 0ull : (~0ull << (shift + 8));
    if (tid < 256) sc.hist[tid] = 0u;
    group_sync<NT, ID>();
    for (int g = 0; g < src.groups(); ++g) {
      const int n = src.count(g);
      for (int i0 = 0; i0 < n; i0 += NT) {   // warp-uniform trip count: the whole warp adds
        const int i = i0 + tid;
        const uint64_t u = i < n ? src.key(g, i) : 0ull;
        warp_hist_add(i < n && (u & hi) == prefix, (uint32_t)(u >> shift) & 255u, sc.hist);
      }
    }
    group_sync<NT, ID>();
    const int c = tid < 256 ? (int)sc.hist[255 - tid] : 0;   // bins in descending order
    int tot;
    const int incl = group_scan_incl<NT, ID>(c, sc.warp_tot, &tot);
    if (tid < 256 && incl - c < remaining && incl >= remaining) {
      sc.found[0] = 255 - tid;
      sc.found[1] = incl - c;
      sc.found[2] = c;
    }
    group_sync<NT, ID>();
    const int d = sc.found[0], above = sc.found[1], in_bin = sc.found[2];
    group_sync<NT, ID>();
    prefix |= (uint64_t)d << shift;
    remaining -= above;
    if (in_bin == remaining || shift == 0) return prefix;
  }
}

// Appends `key` (where `take`) to buf at positions handed out by sc.count, one shared atomic per
// warp.  Lanes may disagree on `take`; the whole warp must call.
__device__ __forceinline__ void warp_append(bool take, uint64_t key, uint64_t* buf, int* counter) {
  const unsigned m = __ballot_sync(0xffffffffu, take);
  if (m == 0u) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (take) buf[base + __popc(m & ((1u << lane) - 1u))] = key;
}

// Keeps the keys >= tau of buf[0..n) (order not kept); returns how many remain.  n <= NT * MAXPER.
template <int NT, int ID, int MAXPER>
__device__ int compact_keys_ge(uint64_t* buf, int n, uint64_t tau, SelScratch<NT>& sc) {
  const int tid = threadIdx.x;
  uint64_t v[MAXPER];
#pragma unroll
  for (int s = 0; s < MAXPER; ++s) {
    const int i = tid + s * NT;
    v[s] = i < n ? buf[i] : 0ull;
  }
  if (tid == 0) sc.count = 0;
  group_sync<NT, ID>();
#pragma unroll
  for (int s = 0; s < MAXPER; ++s) {
    const int i = tid + s * NT;
    warp_append(i < n && v[s] >= tau, v[s], buf, &sc.count);
  }
  group_sync<NT, ID>();
  const int r = sc.count;
  group_sync<NT, ID>();
  return r;
}

}  // namespace lcsa
