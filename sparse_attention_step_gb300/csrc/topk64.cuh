// Top-k (k <= 64) of up to 2048 candidates inside one CTA, by sorting
// networks: each warp bitonic-sorts 64 keys in registers (two per lane), then
// sorted lists of 64 are merged pairwise (the top 64 of two sorted lists is
// the bitonic sequence max(A[i], B[63-i]) followed by a bitonic merge).
//
// Keys are 64-bit: order-preserving score bits in the high word and the
// complement of the block index in the low word, so a larger key means a
// higher score and, between equal scores, the lower block. Key 0 marks an
// empty slot and sorts last.
#pragma once

#include "common.cuh"

namespace msa {

__device__ inline uint64_t sel_key(float score, int block) {
  return (static_cast<uint64_t>(float_to_key(score)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(block));
}
__device__ inline int sel_block(uint64_t key) { return static_cast<int>(~static_cast<uint32_t>(key)); }

__device__ inline uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ inline uint64_t shfl_xor_key(uint64_t v, int m) { return shfl_xor_u64(v, m); }
__device__ inline uint32_t shfl_xor_key(uint32_t v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }

// Sort the warp's 64 keys (x[r] is element 2*lane + r; 64- or 32-bit) in
// descending order.
// The stage loops stay rolled: this runs once or twice per CTA, so a compact
// body that stays in the instruction cache beats straight-line code that is
// fetched cold.
template <typename T>
__device__ inline void warp_sort64_desc(T (&x)[2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int k = 2; k <= 64; k <<= 1) {
    // stages with partner distance j = 2 lj >= 2 pair different lanes
#pragma unroll 1
    for (int lj = k >> 2; lj > 0; lj >>= 1) {
      const bool lower = (lane & lj) == 0;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int e = 2 * lane + r;
        const bool desc = (e & k) == 0;
        const T o = shfl_xor_key(x[r], lj);
        const bool keep_max = (lower == desc);
        x[r] = keep_max ? (x[r] > o ? x[r] : o) : (x[r] < o ? x[r] : o);
      }
    }
    // distance 1: the lane's own pair
    const bool desc = ((2 * lane) & k) == 0;
    const bool swap = desc ? (x[0] < x[1]) : (x[0] > x[1]);
    if (swap) {
      const T t = x[0];
      x[0] = x[1];
      x[1] = t;
    }
  }
}

// Bitonic merge of a warp's 64 keys (element e in lane e/2, slot e%2) that
// form a bitonic sequence: afterwards they are sorted in descending order.
__device__ inline void warp_bitonic_merge64_desc(uint64_t (&x)[2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int lj = 16; lj > 0; lj >>= 1) {
    const bool lower = (lane & lj) == 0;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint64_t o = shfl_xor_u64(x[r], lj);
      x[r] = lower ? (x[r] > o ? x[r] : o) : (x[r] < o ? x[r] : o);
    }
  }
  if (x[0] < x[1]) {
    const uint64_t t = x[0];
    x[0] = x[1];
    x[1] = t;
  }
}

// One warp: out = top 64 of the sorted (descending) lists a and b, sorted.
__device__ inline void warp_merge64(const uint64_t* a, const uint64_t* b, uint64_t* out) {
  const int lane = threadIdx.x & 31;
  uint64_t x[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int e = 2 * lane + r;
    const uint64_t u = a[e], v = b[63 - e];
    x[r] = u > v ? u : v;
  }
  warp_bitonic_merge64_desc(x);
  out[2 * lane] = x[0];
  out[2 * lane + 1] = x[1];
}

// One warp, registers only: a = top 64 of the sorted (descending) lists a and
// b, sorted. Element e of a meets element 63 - e of b, which sits in lane
// 31 - lane (= lane ^ 31), slot 1 - r.
__device__ inline void warp_merge64_reg(uint64_t (&a)[2], const uint64_t (&b)[2]) {
  const uint64_t v0 = shfl_xor_u64(b[1], 31), v1 = shfl_xor_u64(b[0], 31);
  a[0] = a[0] > v0 ? a[0] : v0;
  a[1] = a[1] > v1 ? a[1] : v1;
  warp_bitonic_merge64_desc(a);
}

// Merge `n_lists` sorted lists of 64 keys in buf (a power of two, <= 64) down
// to one; the result is returned (a pointer into buf or tmp). Every thread of
// the CTA calls this; warps take the pairs round-robin.
__device__ inline uint64_t* block_merge_lists(uint64_t* buf, uint64_t* tmp, int n_lists) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  uint64_t* src = buf;
  uint64_t* dst = tmp;
  while (n_lists > 1) {
    const int pairs = n_lists >> 1;
    for (int p = warp; p < pairs; p += nwarps) warp_merge64(src + (2 * p) * 64, src + (2 * p + 1) * 64, dst + p * 64);
    __syncthreads();
    uint64_t* t = src;
    src = dst;
    dst = t;
    n_lists = pairs;
  }
  return src;
}

// block_merge_lists for the first `nwarps` warps of the CTA only: they meet
// at named barrier `bar` (1..15) instead of __syncthreads, so the other warps
// are free meanwhile.
__device__ inline const uint64_t* warps_merge_lists(uint64_t* buf, uint64_t* tmp, int n_lists, int nwarps, int bar) {
  const int warp = threadIdx.x >> 5;
  uint64_t* src = buf;
  uint64_t* dst = tmp;
  while (n_lists > 1) {
    const int pairs = n_lists >> 1;
    for (int p = warp; p < pairs; p += nwarps) warp_merge64(src + (2 * p) * 64, src + (2 * p + 1) * 64, dst + p * 64);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(32 * nwarps) : "memory");
    uint64_t* t = src;
    src = dst;
    dst = t;
    n_lists = pairs;
  }
  return src;
}

// Compare-exchange inside a lane for the 128-key sort: registers r and r ^ j
// (j = 1 or 2), direction from the bitonic block size k.
__device__ inline void lane_stage128(uint64_t (&x)[4], int k, int j) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int p = r ^ j;
    if (p > r) {
      const int e = 4 * lane + r;
      const bool desc = (e & k) == 0;
      const bool swap = desc ? (x[r] < x[p]) : (x[r] > x[p]);
      if (swap) {
        const uint64_t t = x[r];
        x[r] = x[p];
        x[p] = t;
      }
    }
  }
}

// Sort the warp's 128 keys (x[r] is element 4*lane + r) in descending order
// (stage loops rolled, as in warp_sort64_desc).
__device__ inline void warp_sort128_desc(uint64_t (&x)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int k = 2; k <= 128; k <<= 1) {
#pragma unroll 1
    for (int lj = k >> 3; lj > 0; lj >>= 1) {  // partner distance 4 lj >= 4: another lane
      const bool lower = (lane & lj) == 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = 4 * lane + r;
        const bool desc = (e & k) == 0;
        const uint64_t o = shfl_xor_u64(x[r], lj);
        const bool keep_max = (lower == desc);
        x[r] = keep_max ? (x[r] > o ? x[r] : o) : (x[r] < o ? x[r] : o);
      }
    }
    if (k >= 4) lane_stage128(x, k, 2);
    lane_stage128(x, k, 1);
  }
}

// Top-k (k <= 64, 1 <= k <= n) of n <= 4096 keys in shared memory, written
// sorted descending to top[0..64) (entries past k are not meaningful).
// Exact: t = the k-th largest of 64 group maxima is <= the k-th largest key
// (the k best groups each hold a key >= t), so every one of the top k keys is
// >= t. The keys >= t (normally a little over k) are sorted by one warp; if
// more than 128 pass, the keys are sorted in full with the list merge tree.
// `work` holds >= 2 * max(n_pad, 128) + 64 keys; every thread calls this.
__device__ inline void block_topk(const uint64_t* keys, int n, int k, uint64_t* work, uint64_t* top, int* count) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = (n + 63) / 64;  // group size
  uint64_t* gmax = work;        // [64]
  uint64_t* cand = work + 64;   // [128]
  if (tid == 0) *count = 0;
  for (int grp = warp; grp < 64; grp += blockDim.x >> 5) {
    uint64_t m = 0ull;
    for (int i = grp * g + lane; i < min(n, (grp + 1) * g); i += 32) m = keys[i] > m ? keys[i] : m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = shfl_xor_u64(m, off);
      m = o > m ? o : m;
    }
    if (lane == 0) gmax[grp] = m;
  }
  __syncthreads();
  __shared__ uint64_t thr;
  if (warp == 0) {
    uint64_t x[2] = {gmax[2 * lane], gmax[2 * lane + 1]};
    warp_sort64_desc(x);
    // element k-1 of the sorted maxima
    const int e = k - 1;
    const uint64_t mine = (e >> 1) == lane ? x[e & 1] : 0ull;
    uint64_t t = mine;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = shfl_xor_u64(t, off);
      t = o > t ? o : t;
    }
    if (lane == 0) thr = t;
  }
  __syncthreads();
  const uint64_t t = thr;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + tid;
    const bool hit = i < n && keys[i] >= t && keys[i] != 0ull;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    int slot = 0;
    if (lane == 0 && m != 0u) slot = atomicAdd(count, __popc(m));
    slot = __shfl_sync(0xffffffffu, slot, 0);
    const int pos = slot + __popc(m & ((1u << lane) - 1u));
    if (hit && pos < 128) cand[pos] = keys[i];
  }
  __syncthreads();
  const int c = *count;
  if (c <= 128) {
    if (warp == 0) {
      uint64_t x[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = 4 * lane + r;
        x[r] = e < c ? cand[e] : 0ull;
      }
      warp_sort128_desc(x);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = 4 * lane + r;
        if (e < 64) top[e] = x[r];
      }
    }
    __syncthreads();
    return;
  }
  // many keys near the threshold: sort everything in lists of 64 and merge
  int n_lists = 1;
  while (n_lists * 64 < n) n_lists <<= 1;
  uint64_t* a = work;
  uint64_t* b = work + n_lists * 64;
  for (int i = tid; i < n_lists * 64; i += blockDim.x) a[i] = i < n ? keys[i] : 0ull;
  __syncthreads();
  for (int l = warp; l < n_lists; l += blockDim.x >> 5) {
    uint64_t x[2] = {a[l * 64 + 2 * lane], a[l * 64 + 2 * lane + 1]};
    warp_sort64_desc(x);
    a[l * 64 + 2 * lane] = x[0];
    a[l * 64 + 2 * lane + 1] = x[1];
  }
  __syncthreads();
  const uint64_t* best = block_merge_lists(a, b, n_lists);
  for (int i = tid; i < 64; i += blockDim.x) top[i] = best[i];
  __syncthreads();
}

__device__ inline float key_to_float(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Shared scratch of block_select.
struct SelectScratch {
  int hist[1024];
  uint64_t cand[256];
  float wmin[32], wmax[32];
  int n_above, n_cand, bstar, above_bstar;
  float lo, inv;
};

// The k largest (1 <= k <= 64) of n keys in shared memory (0 = empty slot),
// written to out[0..k) in no particular order; returns false (out untouched)
// when the keys crowd too tightly to resolve this way (the caller then falls
// back to block_topk). Exact: scores are binned linearly between their min and
// max into 1024 bins (the bin is non-decreasing in the key); the bin holding
// the k-th largest key is found from the histogram, every key above it is
// kept, and the keys inside it (at most 256) are ranked by pairwise counting.
// Every thread of the CTA calls this.
__device__ inline bool block_select(const uint64_t* keys, int n, int k, uint64_t* out, SelectScratch& sc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nth = blockDim.x;
  // 1. range of the scores
  float mn = INFINITY, mx = -INFINITY;
  for (int i = tid; i < n; i += nth) {
    const uint64_t kk = keys[i];
    if (kk == 0ull) continue;
    const float f = key_to_float(static_cast<uint32_t>(kk >> 32));
    mn = fminf(mn, f);
    mx = fmaxf(mx, f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (lane == 0) {
    sc.wmin[warp] = mn;
    sc.wmax[warp] = mx;
  }
  for (int i = tid; i < 1024; i += nth) sc.hist[i] = 0;
  __syncthreads();
  if (tid == 0) {
    float a = INFINITY, b = -INFINITY;
    for (int w = 0; w < (nth >> 5); ++w) {
      a = fminf(a, sc.wmin[w]);
      b = fmaxf(b, sc.wmax[w]);
    }
    sc.lo = a;
    sc.inv = (b > a) ? 1024.f / (b - a) : 0.f;
    sc.n_above = 0;
    sc.n_cand = 0;
    sc.bstar = -1;
  }
  __syncthreads();
  const float lo = sc.lo, inv = sc.inv;
  auto bin_of = [&](uint64_t kk) {
    const float f = key_to_float(static_cast<uint32_t>(kk >> 32));
    const int b = static_cast<int>((f - lo) * inv);
    return b < 0 ? 0 : (b > 1023 ? 1023 : b);
  };
  // 2. histogram
  for (int i = tid; i < n; i += nth) {
    const uint64_t kk = keys[i];
    if (kk != 0ull) atomicAdd(&sc.hist[bin_of(kk)], 1);
  }
  __syncthreads();
  // 3. the bin of the k-th largest: suffix counts over 4 bins per thread
  {
    int own = 0;
    if (tid < 256)
      for (int j = 0; j < 4; ++j) own += sc.hist[4 * tid + j];
    // inclusive scan over threads (warp shuffles + one pass over warp totals)
    int x = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    __shared__ int wsum[32];
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < (nth >> 5); ++w) {
      if (w < warp) before += wsum[w];
      total += wsum[w];
    }
    int above = total - (before + x);  // keys in bins above this thread's four
    if (tid < 256 && above < k && above + own >= k) {
      for (int j = 3; j >= 0; --j) {
        const int b = 4 * tid + j;
        if (above + sc.hist[b] >= k) {
          sc.bstar = b;
          sc.above_bstar = above;
          break;
        }
        above += sc.hist[b];
      }
    }
    __syncthreads();
  }
  const int bstar = sc.bstar;
  if (bstar < 0 || sc.hist[bstar] > 256) return false;  // uniform decision: shared values
  const int need = k - sc.above_bstar;
  // 4. keep the keys above the bin; gather the bin's keys
  for (int i = tid; i < n; i += nth) {
    const uint64_t kk = keys[i];
    if (kk == 0ull) continue;
    const int b = bin_of(kk);
    if (b > bstar) out[atomicAdd(&sc.n_above, 1)] = kk;
    else if (b == bstar) sc.cand[atomicAdd(&sc.n_cand, 1)] = kk;
  }
  __syncthreads();
  // 5. rank inside the bin (keys are distinct: they carry the block index)
  const int nc = sc.n_cand, base = sc.n_above;
  for (int i = tid; i < nc; i += nth) {
    const uint64_t me = sc.cand[i];
    int rank = 0;
    for (int j = 0; j < nc; ++j) rank += sc.cand[j] > me;
    if (rank < need) out[base + rank] = me;
  }
  __syncthreads();
  return true;
}

// Shared scratch of block_kth_largest.
struct RadixScratch {
  uint32_t hist[256];
  uint64_t bin_keys[32];
  uint64_t prefix, mask, kth;
  int need, done, n_bin;
};

// The kk-th largest (kk >= 1) of the nonzero keys in keys[0..n) (nonzero keys
// are distinct: they carry the block index), or 1 when fewer than kk keys are
// nonzero (every nonzero key is >= 1). A most-significant-digit radix select:
// each pass counts, among the keys that share the digits fixed so far, the
// next 8-bit digit (lanes with the same digit add their count with one atomic,
// so a crowded digit costs one atomic per warp), and one warp finds the digit
// that holds the kk-th key. Once that digit holds at most 32 keys they are
// gathered and ranked by pairwise counting. Typical scores need two passes.
// Every thread of the CTA calls this (it uses __syncthreads).
__device__ inline uint64_t block_kth_largest(const uint64_t* keys, int n, int kk, RadixScratch& rs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nth = blockDim.x;
  if (tid == 0) {
    rs.prefix = 0ull;
    rs.mask = 0ull;
    rs.need = kk;
    rs.done = 0;
    rs.kth = 1ull;
  }
  for (int shift = 56;; shift -= 8) {
    for (int i = tid; i < 256; i += nth) rs.hist[i] = 0u;
    __syncthreads();
    const uint64_t prefix = rs.prefix, mask = rs.mask;
    for (int base = 0; base < n; base += nth) {
      const int i = base + tid;
      const uint64_t key = i < n ? keys[i] : 0ull;
      const bool in = key != 0ull && (key & mask) == prefix;
      const int digit = in ? static_cast<int>((key >> shift) & 255u) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (in && (__ffs(peers) - 1) == lane) atomicAdd(&rs.hist[digit], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 255 - 8 l - j, j = 0..7 (descending over the warp)
      uint32_t h[8], sum = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = rs.hist[255 - 8 * lane - j];
        sum += h[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      const uint32_t need = static_cast<uint32_t>(rs.need);
      if (total < need) {
        // fewer keys than kk (only possible in the first pass): all are kept
        if (lane == 0) rs.done = 1;
      } else {
        uint32_t above = incl - sum;
        if (above < need && incl >= need) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (above + h[j] >= need) {
              const int d = 255 - 8 * lane - j;
              rs.prefix = prefix | (static_cast<uint64_t>(d) << shift);
              rs.mask = mask | (0xFFull << shift);
              rs.need = static_cast<int>(need - above);
              if (h[j] <= 32u || shift == 0) {
                rs.done = 2;
                rs.n_bin = 0;
              }
              break;
            }
            above += h[j];
          }
        }
      }
    }
    __syncthreads();
    if (rs.done != 0) break;
  }
  if (rs.done == 2) {
    const uint64_t prefix = rs.prefix, mask = rs.mask;
    for (int i = tid; i < n; i += nth) {
      const uint64_t key = keys[i];
      if (key != 0ull && (key & mask) == prefix) {
        const int slot = atomicAdd(&rs.n_bin, 1);
        if (slot < 32) rs.bin_keys[slot] = key;
      }
    }
    __syncthreads();
    if (warp == 0) {
      const int nb = min(rs.n_bin, 32);
      const uint64_t me = lane < nb ? rs.bin_keys[lane] : 0ull;
      int rank = 0;
      for (int j = 0; j < nb; ++j) rank += rs.bin_keys[j] > me ? 1 : 0;
      if (lane < nb && rank == rs.need - 1) rs.kth = me;
    }
    __syncthreads();
  }
  return rs.kth;
}

// Append every nonzero key >= t of keys[0..n) to out (order unspecified) and
// return how many there are. `count` is a shared counter; every thread of the
// CTA calls this (it uses __syncthreads).
__device__ inline int block_compact_ge(const uint64_t* keys, int n, uint64_t t, uint64_t* out, int cap, int* count) {
  const int tid = threadIdx.x, lane = tid & 31, nth = blockDim.x;
  if (tid == 0) *count = 0;
  __syncthreads();
  for (int base = 0; base < n; base += nth) {
    const int i = base + tid;
    const uint64_t key = i < n ? keys[i] : 0ull;
    const bool hit = key != 0ull && key >= t;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    int slot = 0;
    if (lane == 0 && m != 0u) slot = atomicAdd(count, __popc(m));
    slot = __shfl_sync(0xffffffffu, slot, 0);
    const int pos = slot + __popc(m & ((1u << lane) - 1u));
    if (hit && pos < cap) out[pos] = key;
  }
  __syncthreads();
  return min(*count, cap);
}

}  // namespace msa
