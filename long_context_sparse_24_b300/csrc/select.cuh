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

// The outcome of a selection: the keys at or above tau are taken, `count` of them.
struct SelResult {
  uint64_t tau;
  int count;
};

// Most-significant-digit radix selection over the keys of buf[0..n) at or above lo (shared memory,
// unique keys; with fewer than k of them at or above lo, all of those: {lo, their count}):
// BITS-bit digits, the first one ending at the highest bit in which the largest and the smallest
// key differ (the leading bits every key shares need no pass).  A level counts the keys under the
// current prefix per digit value, finds the digit bin that holds the k-th largest key and stops
// once the keys at or above that bin's lower edge number at most k + slack; else the bin becomes
// the prefix of the next level.  slack = 0 gives the exact selection (count == k); with unique
// keys the last level's bins hold one key each, so the loop ends there at the latest.  hist: 1 <<
// BITS counters of shared memory, left at zero.
template <int NT, int ID, int BITS>
__device__ SelResult select_top(const uint64_t* buf, int n, int k, int slack, SelScratch<NT>& sc, uint32_t* hist,
                                uint64_t lo = 0ull) {
  constexpr int B = 1 << BITS;
  constexpr int kBatch = 8;
  constexpr int PER = (B + NT - 1) / NT;   // bins a thread scans, in descending order
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long kmax = 0ull, kmin = ~0ull;
  for (int i = tid; i < n; i += NT) {
    const unsigned long long u = buf[i];
    if (u < lo) continue;
    kmax = u > kmax ? u : kmax;
    kmin = u < kmin ? u : kmin;
  }
  for (int i = tid; i < B; i += NT) hist[i] = 0u;
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
  group_sync<NT, ID>();   // (span is free again for the caller)
  if (kmax < kmin) return SelResult{lo, 0};      // no key at or above lo
  if (kmax == kmin) return SelResult{k <= 1 ? kmax : lo, 1};   // one key: the k-th largest, or fewer than k
  const int hb = 63 - __clzll((long long)(kmax ^ kmin));   // the highest bit in which keys differ
  int width = hb + 1 < BITS ? hb + 1 : BITS;
  int shift = hb + 1 - width;
  uint64_t prefix = hb >= 63 ? 0ull : (kmax & (~0ull << (hb + 1)));
  int above0 = 0;   // keys above the current prefix's range
  for (;;) {
    const uint64_t hi_mask = shift + width >= 64 ? 0ull : (~0ull << (shift + width));
    const uint32_t dmask = (1u << width) - 1u;
    // a thread's keys are read kBatch at a time before any counter is touched, so that their
    // loads overlap (a load of buf cannot be moved above an atomic on hist: both are shared memory)
    for (int i0 = tid; i0 < n; i0 += NT * kBatch) {
      uint64_t v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) v[u] = i0 + u * NT < n ? buf[i0 + u * NT] : 0ull;
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (i0 + u * NT < n && v[u] >= lo && (v[u] & hi_mask) == prefix)
          atomicAdd(&hist[(uint32_t)(v[u] >> shift) & dmask], 1u);
    }
    group_sync<NT, ID>();
    // thread t scans bins B-1-t*PER down to B-(t+1)*PER
    int c = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int pos = tid * PER + j;
      c += pos < B ? (int)hist[B - 1 - pos] : 0;
    }
    int tot;
    const int incl = group_scan_incl<NT, ID>(c, sc.warp_tot, &tot);
    if (above0 + tot < k) {   // (first level only: every key at or above lo is taken)
      for (int i = tid; i < B; i += NT) hist[i] = 0u;
      group_sync<NT, ID>();
      return SelResult{lo, above0 + tot};
    }
    if (incl - c + above0 < k && incl + above0 >= k) {
      int cum = above0 + incl - c;
      for (int j = 0; j < PER; ++j) {
        const int pos = tid * PER + j;
        const int h = pos < B ? (int)hist[B - 1 - pos] : 0;
        if (cum + h >= k) {
          sc.found[0] = B - 1 - pos;
          sc.found[1] = cum;
          sc.found[2] = h;
          break;
        }
        cum += h;
      }
    }
    group_sync<NT, ID>();
    const int d = sc.found[0], above = sc.found[1], in_bin = sc.found[2];
    for (int i = tid; i < B; i += NT) hist[i] = 0u;
    group_sync<NT, ID>();
    prefix |= (uint64_t)d << shift;
    if (above + in_bin <= k + slack || shift == 0) return SelResult{prefix, above + in_bin};
    above0 = above;
    width = shift < BITS ? shift : BITS;
    shift -= width;
  }
}

// The threshold tau with exactly k of buf[0..n)'s keys >= tau (k <= n; keys unique); keys below
// lo are left out (at least k keys at or above it).
template <int NT, int ID, int BITS>
__device__ __forceinline__ uint64_t kth_largest_key(const uint64_t* buf, int n, int k, SelScratch<NT>& sc,
                                                    uint32_t* hist, uint64_t lo = 0ull) {
  return select_top<NT, ID, BITS>(buf, n, k, 0, sc, hist, lo).tau;
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

// Keeps the keys >= tau of buf[0..n) (order not kept); returns how many remain.  The keys go in
// blocks of NT * MAXPER: a block is read into registers, a prefix sum over the group gives every
// thread the place of its kept keys, and the writes start once the whole block has been read (the
// scan's barriers); a kept key lands below the end of its own block (no more keys are kept than
// were read), so it only overwrites keys already read.
template <int NT, int ID, int MAXPER>
__device__ int compact_keys_ge(uint64_t* buf, int n, uint64_t tau, SelScratch<NT>& sc) {
  const int tid = threadIdx.x;
  int kept = 0;   // (the same on every thread)
  for (int b0 = 0; b0 < n; b0 += NT * MAXPER) {
    uint64_t v[MAXPER];
    int mine = 0;
#pragma unroll
    for (int s = 0; s < MAXPER; ++s) {
      const int i = b0 + tid + s * NT;
      v[s] = i < n ? buf[i] : 0ull;
      mine += i < n && v[s] >= tau ? 1 : 0;
    }
    int tot;
    int pos = kept + group_scan_incl<NT, ID>(mine, sc.warp_tot, &tot) - mine;
#pragma unroll
    for (int s = 0; s < MAXPER; ++s)
      if (b0 + tid + s * NT < n && v[s] >= tau) buf[pos++] = v[s];
    kept += tot;
  }
  group_sync<NT, ID>();
  return kept;
}

}  // namespace lcsa
