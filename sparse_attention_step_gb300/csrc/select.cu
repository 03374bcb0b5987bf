// Step 1b/1c: group index query, block scores and top-k block selection
// ("MiniMax goes sparse", §1 Step 1: one index query per GQA group, block-level
// scores, TopK keeps the best KV blocks per layer and group; §3: in prefill
// the index branch still scans the whole input).
//
// Three kernels:
//   qidx_prefill_kernel  q_idx of a 64-token prefill tile = sum over its tokens
//                        and the group's heads (fp32, token-major order).
//   score_kernel         streams the pooled keys of each unit once (bandwidth
//                        bound, 16-byte loads, one half-warp per block row) and
//                        writes fp32 scores; for decode it forms q_idx inline
//                        from the G query heads.
//   topk_kernel          per unit, radix select of the k-th largest score in
//                        shared memory (4 passes of 8-bit digits over
//                        order-preserving keys), ties to the lower block, then
//                        an ordered compaction that emits the kept blocks in
//                        ascending order followed by the forced block.
#include <float.h>

#include "kernels.cuh"

namespace msa {

// ---------------------------------------------------------------------------
// q_idx for prefill tiles. grid (Hkv, n_tiles), 128 threads (one per dim).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) qidx_prefill_kernel(const T* __restrict__ q, int hq, int hkv,
                                                          int n_q_tokens, float* __restrict__ qidx) {
  const int h = blockIdx.x;
  const int tile = blockIdx.y;
  const int d = threadIdx.x;
  const int grp = hq / hkv;
  const int r0 = tile * kBlock;
  const int r1 = min(n_q_tokens, r0 + kBlock);
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) {
    const T* row = q + (static_cast<int64_t>(r) * hq + h * grp) * kHeadDim + d;
    for (int g = 0; g < grp; ++g) acc += static_cast<float>(row[g * kHeadDim]);
  }
  qidx[(static_cast<int64_t>(tile) * hkv + h) * kHeadDim + d] = acc;
}

// ---------------------------------------------------------------------------
// Block scores.
// Decode:  grid (chunks, Hkv, batch); unit = s*Hkv + h; q_idx from q inline.
// Prefill: grid (chunks, Hkv, ceil(n_tiles / kTiles)); unit = tile*Hkv + h;
//          q_idx from the workspace; each pooled row is scored against
//          kTiles tiles so it is read once per kTiles tiles.
// Scores of non-candidates in the chunk are written as -inf.
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kScoreChunk = 256;  // pooled rows per CTA

template <typename T>
__device__ inline void load8(const T* p, float (&x)[8]);
template <>
__device__ inline void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
  uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <>
__device__ inline void load8<float>(const float* p, float (&x)[8]) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

struct ScoreArgs {
  int hq, hkv;
  int prefill;        // 0 decode, 1 prefill
  int force_local;
  int64_t q_start;    // prefill
  int n_tiles;        // prefill
  int64_t max_blocks; // row stride of the score array
};

template <typename T, int kTiles>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const T* __restrict__ q, const float* __restrict__ qidx_ws,
                                                             const T* __restrict__ pooled, KvView kv, ScoreArgs a,
                                                             float* __restrict__ scores, int32_t* status) {
  const int h = blockIdx.y;
  const int e = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
  const int64_t chunk0 = static_cast<int64_t>(blockIdx.x) * kScoreChunk;

  float qi[kTiles][8];
  int64_t n_cand[kTiles];
  int64_t unit[kTiles];
  int seq = 0;
  if (!a.prefill) {
    seq = blockIdx.z;
    const int grp = a.hq / a.hkv;
    const int64_t len = kv.seq_len(seq, status, kIdScore);
    const int64_t nb = (len + kBlock - 1) / kBlock;
    const int64_t nbf = len / kBlock;
    n_cand[0] = a.force_local ? min(nbf, nb - 1) : nbf;
    if (n_cand[0] < 0) n_cand[0] = 0;
    unit[0] = static_cast<int64_t>(seq) * a.hkv + h;
#pragma unroll
    for (int i = 0; i < 8; ++i) qi[0][i] = 0.f;
    for (int g = 0; g < grp; ++g) {
      float x[8];
      load8<T>(q + (static_cast<int64_t>(seq) * a.hq + h * grp + g) * kHeadDim + 8 * e, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) qi[0][i] += x[i];
    }
  } else {
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      const int tile = blockIdx.z * kTiles + t;
      const bool live = tile < a.n_tiles;
      n_cand[t] = live ? a.q_start / kBlock + tile : 0;
      unit[t] = static_cast<int64_t>(live ? tile : 0) * a.hkv + h;
      if (live) {
        float4 u = *reinterpret_cast<const float4*>(qidx_ws + unit[t] * kHeadDim + 8 * e);
        float4 v = *reinterpret_cast<const float4*>(qidx_ws + unit[t] * kHeadDim + 8 * e + 4);
        qi[t][0] = u.x; qi[t][1] = u.y; qi[t][2] = u.z; qi[t][3] = u.w;
        qi[t][4] = v.x; qi[t][5] = v.y; qi[t][6] = v.z; qi[t][7] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) qi[t][i] = 0.f;
      }
    }
  }
  int64_t n_max = 0;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) n_max = max(n_max, n_cand[t]);
  const int64_t row_end = min(chunk0 + kScoreChunk, a.max_blocks);

  constexpr int kRowsPerIter = kScoreThreads / 16;
  constexpr int kUnroll = 4;
#pragma unroll 1
  for (int64_t r0 = chunk0; r0 < row_end; r0 += kRowsPerIter * kUnroll) {
    float kp[kUnroll][8];
    bool have[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t b = r0 + u * kRowsPerIter + hw;
      have[u] = b < n_max && b < row_end;
      if (have[u]) {
        const int64_t prow = kv.pooled_row(seq, h, b, status, kIdScore);
        if (prow < 0) {
          have[u] = false;
        } else {
          load8<T>(pooled + prow * kHeadDim + 8 * e, kp[u]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t b = r0 + u * kRowsPerIter + hw;
      const bool in_range = b < row_end;  // all lanes still join the shuffles
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        float part = 0.f;
        if (have[u]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) part = fmaf(qi[t][i], kp[u][i], part);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 8);
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        if (e == 0 && in_range && (!a.prefill || blockIdx.z * kTiles + t < a.n_tiles)) {
          scores[unit[t] * a.max_blocks + b] = (b < n_cand[t] && have[u]) ? part : -INFINITY;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Top-k. grid (Hkv, outer) with outer = batch (decode) or n_tiles (prefill).
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;

// Inclusive block-wide scan of one int per thread; returns the inclusive
// value; *total gets the block sum. Uses `tmp` (>= 33 ints of shared memory).
__device__ inline int block_inclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < nw) tmp[lane] = w;
    if (lane == 31) tmp[32] = w;
  }
  __syncthreads();
  const int res = x + (warp > 0 ? tmp[warp - 1] : 0);
  *total = tmp[32];
  __syncthreads();
  return res;
}

struct TopkArgs {
  int hkv;
  int prefill;
  int force_local;
  int k_scored;
  int k_total;
  int64_t q_start;
  int64_t max_blocks;
};

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, KvView kv, TopkArgs a,
                                                           int32_t* __restrict__ idx_out, int32_t* status) {
  extern __shared__ uint32_t keys[];  // [max_blocks]
  __shared__ int hist[256];
  __shared__ int scan_tmp[33];
  __shared__ int sel_digit, sel_above;

  const int h = blockIdx.x;
  const int outer = blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t unit = static_cast<int64_t>(outer) * a.hkv + h;

  int64_t n, forced;
  if (!a.prefill) {
    const int64_t len = kv.seq_len(outer, status, kIdTopk);
    const int64_t nb = (len + kBlock - 1) / kBlock;
    const int64_t nbf = len / kBlock;
    n = a.force_local ? min(nbf, nb - 1) : nbf;
    forced = (a.force_local && nb > 0) ? nb - 1 : -1;
  } else {
    n = a.q_start / kBlock + outer;
    forced = a.force_local ? n : -1;
  }
  if (n < 0) n = 0;
  const int k = static_cast<int>(min(static_cast<int64_t>(a.k_scored), n));
  const float* sc = scores + unit * a.max_blocks;
  int32_t* out = idx_out + unit * a.k_total;

  uint32_t thresh = 0;  // keys >= thresh ... (see below)
  int take_equal = 0;   // how many keys == thresh to keep (lowest indices)
  const bool all = (k >= n);
  if (!all && k > 0) {
    for (int64_t i = tid; i < n; i += blockDim.x) keys[i] = float_to_key(sc[i]);
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < n; i += blockDim.x) {
        const uint32_t key = keys[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns digits [8l, 8l+8); suffix sums from the top digit down
        int own = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) own += hist[8 * tid + j];
        int suf = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          int y = __shfl_down_sync(0xffffffffu, suf, off);
          if (tid + off < 32) suf += y;
        }
        const int above_lane = suf - own;  // count in lanes > tid
        if (above_lane < remaining && suf >= remaining) {
          int acc = above_lane;
          for (int d = 8 * tid + 7; d >= 8 * tid; --d) {
            if (acc + hist[d] >= remaining) {
              sel_digit = d;
              sel_above = acc;
              break;
            }
            acc += hist[d];
          }
        }
      }
      __syncthreads();
      remaining -= sel_above;
      prefix |= static_cast<uint32_t>(sel_digit) << shift;
      mask |= 255u << shift;
      __syncthreads();
    }
    thresh = prefix;
    take_equal = remaining;
  }

  // Ordered compaction over contiguous per-thread ranges.
  const int64_t per = (n + blockDim.x - 1) / blockDim.x;
  const int64_t lo = min(n, static_cast<int64_t>(tid) * per);
  const int64_t hi = min(n, lo + per);
  int written = 0;
  if (k > 0) {
    int eq_before = 0;
    if (!all) {
      int my_eq = 0;
      for (int64_t i = lo; i < hi; ++i) my_eq += keys[i] == thresh;
      int tot;
      eq_before = block_inclusive_scan(my_eq, scan_tmp, &tot) - my_eq;
    }
    int my_sel = 0;
    {
      int eq = eq_before;
      for (int64_t i = lo; i < hi; ++i) {
        if (all) {
          ++my_sel;
        } else {
          const uint32_t key = keys[i];
          if (key > thresh) ++my_sel;
          else if (key == thresh && eq++ < take_equal) ++my_sel;
        }
      }
    }
    int tot;
    int pos = block_inclusive_scan(my_sel, scan_tmp, &tot) - my_sel;
    {
      int eq = eq_before;
      for (int64_t i = lo; i < hi; ++i) {
        bool keep;
        if (all) {
          keep = true;
        } else {
          const uint32_t key = keys[i];
          keep = key > thresh || (key == thresh && eq++ < take_equal);
        }
        if (keep) out[pos++] = static_cast<int32_t>(i);
      }
    }
    written = tot;
  }
  if (tid == 0) {
    int w = written;
    if (forced >= 0) out[w++] = static_cast<int32_t>(forced);
    for (; w < a.k_total; ++w) out[w] = -1;
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename T>
cudaError_t launch_select(const T* q, int hq, int n_q_tokens, const T* pooled, const KvView& kv, int batch,
                          const msa_select_cfg& cfg, int32_t* idx_out, int k_total, float* scores, float* qidx_ws,
                          int32_t* status, cudaStream_t stream) {
  const int prefill = cfg.q_tile == kBlock;
  const int64_t max_blocks = kv.max_blocks();
  ScoreArgs sa{hq, kv.hkv, prefill, cfg.force_local, cfg.q_start, 0, max_blocks};
  const unsigned chunks = static_cast<unsigned>((max_blocks + kScoreChunk - 1) / kScoreChunk);
  int outer;
  if (!prefill) {
    outer = batch;
    score_kernel<T, 1><<<dim3(chunks, kv.hkv, batch), kScoreThreads, 0, stream>>>(q, nullptr, pooled, kv, sa,
                                                                                  scores, status);
  } else {
    const int n_tiles = (n_q_tokens + kBlock - 1) / kBlock;
    outer = n_tiles;
    sa.n_tiles = n_tiles;
    qidx_prefill_kernel<T><<<dim3(kv.hkv, n_tiles), 128, 0, stream>>>(q, hq, kv.hkv, n_q_tokens, qidx_ws);
    constexpr int kT = 8;
    // only the chunks below the last tile's diagonal hold candidates
    const int64_t last = cfg.q_start / kBlock + n_tiles;
    const unsigned pchunks = static_cast<unsigned>((min(last, max_blocks) + kScoreChunk - 1) / kScoreChunk);
    score_kernel<T, kT><<<dim3(pchunks, kv.hkv, (n_tiles + kT - 1) / kT), kScoreThreads, 0, stream>>>(
        q, qidx_ws, pooled, kv, sa, scores, status);
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  TopkArgs ta{kv.hkv, prefill, cfg.force_local, cfg.k_scored, k_total, cfg.q_start, max_blocks};
  const size_t smem = static_cast<size_t>(max_blocks) * sizeof(uint32_t);
  topk_kernel<<<dim3(kv.hkv, outer), kTopkThreads, smem, stream>>>(scores, kv, ta, idx_out, status);
  return cudaGetLastError();
}

cudaError_t set_topk_smem(size_t bytes) {
  return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template cudaError_t launch_select<__nv_bfloat16>(const __nv_bfloat16*, int, int, const __nv_bfloat16*,
                                                  const KvView&, int, const msa_select_cfg&, int32_t*, int, float*,
                                                  float*, int32_t*, cudaStream_t);
template cudaError_t launch_select<float>(const float*, int, int, const float*, const KvView&, int,
                                          const msa_select_cfg&, int32_t*, int, float*, float*, int32_t*,
                                          cudaStream_t);

}  // namespace msa
