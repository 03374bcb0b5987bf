// Step 1b/1c: group index query, block scores and top-k block selection
// ("MiniMax goes sparse", §1 Step 1: one index query per GQA group, block-level
// scores, TopK keeps the best KV blocks per layer and group; §3: in prefill
// the index branch still scans the whole input).
//
// Kernels:
//   qidx_prefill_kernel  q_idx of a 64-token prefill tile = sum over its tokens
//                        and the group's heads (fp32).
//   score_kernel         streams the summary keys of each unit once (16-byte
//                        loads, one half-warp per block row) and writes fp32
//                        scores; for decode it forms q_idx inline from the G
//                        query heads. bf16 prefill uses score_prefill_mma_kernel
//                        (tensor cores, 8 tiles per summary row read).
//   topk_kernel          per unit: a shared-memory histogram of the top 12
//                        bits of the order-preserving score keys gives the bin
//                        that holds the k-th largest score; the scores in that
//                        bin are refined by two 10-bit radix passes, ties go
//                        to the lower block, and an ordered compaction emits
//                        the kept blocks ascending, then the forced block.
// The decode selection for k <= 64 is select_decode_kernel (below).
#include <float.h>

#include "kernels.cuh"
#include "rows.cuh"
#include "topk64.cuh"

namespace msa {

// ---------------------------------------------------------------------------
// q_idx for prefill tiles. grid (Hkv, n_tiles), 256 threads: the tile's
// 64 tokens x G heads rows are split over 16 row slots (16 lanes each reading
// one 256-byte row with 16-byte loads, 8 rows in flight per thread), and the
// 16 partial sums of each dim are added in slot order through shared memory.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) qidx_prefill_kernel(const T* __restrict__ q, int hq, int hkv,
                                                          const PrefillBatch pb, float* __restrict__ qidx) {
  __shared__ float part[16][kHeadDim + 4];
  const int h = blockIdx.x;
  const int tile = blockIdx.y;  // global tile
  const int e = threadIdx.x & 15, slot = threadIdx.x >> 4;
  const int grp = hq / hkv;
  const int s = pb.seq_of_tile(tile);
  const int j0 = max(pb.tile_row0(s, tile), 0);                                       // the tile's first token
  const int r0 = pb.q_off[s] + j0;                                                    // its row in q
  const int n_rows = (min(pb.q_cnt[s], pb.tile_row0(s, tile) + kBlock) - j0) * grp;  // token-major, head-minor
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int i0 = slot; i0 < n_rows; i0 += 16 * 8) {
    RawRow<T> x[8];  // raw 16-byte pieces: few registers per row in flight
    bool have[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 16 * u;
      have[u] = i < n_rows;
      if (have[u]) x[u].load(q + (static_cast<int64_t>(r0 + i / grp) * hq + h * grp + i % grp) * kHeadDim + 8 * e);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (have[u]) x[u].add_to(acc);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[slot][8 * e + j] = acc[j];
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) t += part[k][threadIdx.x];
    qidx[(static_cast<int64_t>(tile) * hkv + h) * kHeadDim + threadIdx.x] = t;
  }
}

// bf16 q: the tile's rows (64 tokens x G heads, 256 bytes each; a token's G
// heads are contiguous) are pulled into shared memory with 16-byte cp.async in
// chunks of 64 rows through a 4-stage ring (three chunks in flight while one
// is summed, three CTAs per SM), then summed like the kernel above: 16 row
// slots per 16-byte piece of the dims, each slot's rows in ascending order,
// the slots' partial sums added in slot order. grid (Hkv, n_tiles), 256
// threads, dynamic shared memory kQidxStages x 16 KB.
constexpr int kQidxThreads = 256;
constexpr int kQidxChunkRows = 64;  // 16 KB of rows per chunk
constexpr int kQidxStages = 4;
__global__ void __launch_bounds__(kQidxThreads) qidx_prefill_bf16_kernel(const __nv_bfloat16* __restrict__ q, int hq,
                                                                       int hkv, const PrefillBatch pb,
                                                                       float* __restrict__ qidx) {
  extern __shared__ __align__(16) uint8_t qrows[];  // [kQidxStages][kQidxChunkRows][256 B]
  __shared__ float part[16][kHeadDim + 4];
  const int h = blockIdx.x;
  const int tile = blockIdx.y;  // global tile
  const int grp = hq / hkv;
  const int s = pb.seq_of_tile(tile);
  const int j0 = max(pb.tile_row0(s, tile), 0);  // the tile's first token within its sequence's chunk
  const int r0 = pb.q_off[s] + j0;
  const int n_rows = (min(pb.q_cnt[s], pb.tile_row0(s, tile) + kBlock) - j0) * grp;  // token-major, head-minor
  const int n_ch = (n_rows + kQidxChunkRows - 1) / kQidxChunkRows;
  const int tid = threadIdx.x;
  // chunk c (rows [64 c, 64 c + 64)) into stage c mod kQidxStages; one commit
  // group per call, empty past the last chunk, so the wait count is uniform
  auto issue = [&](int c) {
    if (c < n_ch) {
      uint8_t* stage = qrows + (c % kQidxStages) * (kQidxChunkRows * 256);
      const int rows = min(kQidxChunkRows, n_rows - c * kQidxChunkRows);
      for (int i = tid; i < rows * 16; i += kQidxThreads) {
        const int lr = i >> 4, pc = i & 15;
        const int row = c * kQidxChunkRows + lr;
        const int t = row / grp, g = row - t * grp;
        cp_async16(stage + lr * 256 + pc * 16, q + (static_cast<int64_t>(r0 + t) * hq + h * grp + g) * kHeadDim + 8 * pc);
      }
    }
    cp_async_commit();
  };
  for (int c = 0; c < kQidxStages - 1; ++c) issue(c);
  const int e = tid & 15, slot = tid >> 4;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int c = 0; c < n_ch; ++c) {
    cp_async_wait<kQidxStages - 2>();  // chunk c has landed (this thread's pieces)
    __syncthreads();                   // every thread's pieces; chunk c - 1's stage is free again
    issue(c + kQidxStages - 1);
    const uint8_t* stage = qrows + (c % kQidxStages) * (kQidxChunkRows * 256);
    const int rows = min(kQidxChunkRows, n_rows - c * kQidxChunkRows);
#pragma unroll 4
    for (int lr = slot; lr < rows; lr += 16) {  // 64 rows per chunk: each slot's rows stay ascending
      RawRow<__nv_bfloat16> x;
      x.w = *reinterpret_cast<const uint4*>(stage + lr * 256 + 16 * e);
      x.add_to(acc);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[slot][8 * e + j] = acc[j];
  __syncthreads();
  if (tid < kHeadDim) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) t += part[k][tid];
    qidx[(static_cast<int64_t>(tile) * hkv + h) * kHeadDim + tid] = t;
  }
}
constexpr size_t kQidxSmemMax = static_cast<size_t>(kQidxStages) * kQidxChunkRows * 256;

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
constexpr int kHistBits = 12;     // first radix digit of the top-k: top 12 bits of the score key
constexpr int kHistBins = 1 << kHistBits;

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
    n_cand[0] = (a.force_local & kForceLocal) ? min(nbf, nb - 1) : nbf;
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
  constexpr int kUnroll = kScoreChunk / kRowsPerIter;  // every row of the chunk in flight at once
#pragma unroll 1
  for (int64_t r0 = chunk0; r0 < row_end; r0 += kRowsPerIter * kUnroll) {
    RawRow<T> kp[kUnroll];
    bool have[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t b = r0 + u * kRowsPerIter + hw;
      have[u] = b < n_max && b < row_end;
      if (have[u]) {
        kp[u].load(pooled + kv.pooled_row(seq, h, b) * kHeadDim + 8 * e);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t b = r0 + u * kRowsPerIter + hw;
      const bool in_range = b < row_end;  // all lanes still join the shuffles
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        float part = have[u] ? kp[u].dot(qi[t]) : 0.f;
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
// Prefill block scores on the tensor cores (bf16 summaries).
// grid (ceil(rows / 128), Hkv, ceil(n_tiles / 16)), 256 threads. The CTA
// copies 128 summary rows into shared memory with cp.async (128-byte swizzle,
// two 64-dim halves) and each warp scores 16 of them against the index queries
// of 16 tiles at once: mma.sync with the tiles as the N columns (two n-tiles
// of 8), the fp32 index queries split into a bf16 head and a bf16 remainder.
// The 16 index queries are read once per CTA (coalesced) into shared memory,
// where every warp takes its operand fragments.
// ---------------------------------------------------------------------------
constexpr int kPsRows = 128;
constexpr int kPsTiles = 16;

__global__ void __launch_bounds__(256) score_prefill_mma_kernel(const float* __restrict__ qidx_ws,
                                                                const __nv_bfloat16* __restrict__ pooled,
                                                                KvView kv, ScoreArgs a, const PrefillBatch pb,
                                                                float* __restrict__ scores, int32_t* status) {
  __shared__ __align__(1024) uint8_t rows_s[kPsRows * kHeadDim * 2];
  __shared__ __align__(16) float qs[kPsTiles][kHeadDim + 8];  // padded: conflict-free 8-byte fragment reads
  const int h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // 16 tiles of one sequence: global tiles t0 .. t_end - 1, local tiles j0 ..
  const int seq = pb.seq_of_group(blockIdx.z);
  const int j0 = (blockIdx.z - pb.grp_off[seq]) * kPsTiles;
  const int t0 = pb.tile_off[seq] + j0;
  const int t_end = min(t0 + kPsTiles, pb.tile_off[seq + 1]);
  const int64_t diag0 = pb.q_start[seq] / kBlock + j0;  // candidates of tile t0 + t: blocks < diag0 + t
  const int64_t chunk0 = static_cast<int64_t>(blockIdx.x) * kPsRows;
  int64_t n_max = 0;
  for (int t = 0; t < kPsTiles; ++t)
    if (t0 + t < t_end) n_max = max(n_max, diag0 + t);
  const int64_t row_end = min(chunk0 + kPsRows, a.max_blocks);
  // cp.async: 128 rows x 16 pieces of 16 bytes, 8 per thread
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int j = tid + 256 * u;
    const int row = j >> 4, pc = j & 15;
    const int64_t b = chunk0 + row;
    if (b < n_max && b < row_end)
      cp_async16(rows_s + (pc >> 3) * (kPsRows * 128) + row * 128 + (((pc & 7) ^ (row & 7)) << 4),
                 pooled + kv.pooled_row(seq, h, b) * kHeadDim + 8 * pc);
  }
  cp_async_commit();
#pragma unroll
  for (int u = 0; u < kPsTiles / 8; ++u) {
    // the 16 tiles' index queries (zeros past the last tile), one float4 a thread each time
    const int tt = 8 * u + (tid >> 5), d4 = tid & 31;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t0 + tt < t_end)
      x = reinterpret_cast<const float4*>(qidx_ws + (static_cast<int64_t>(t0 + tt) * a.hkv + h) * kHeadDim)[d4];
    *reinterpret_cast<float4*>(&qs[tt][4 * d4]) = x;
  }
  cp_async_wait<0>();
  __syncthreads();
  const uint32_t sbase = smem_u32(rows_s);
  const int krow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int kchunk = lane >> 4;
  const int g = lane >> 2, c = lane & 3;
  // one n-tile of 8 tiles at a time; B operands: column g = tile t0 + 8 nt + g
#pragma unroll 1
  for (int nt = 0; nt < kPsTiles / 8; ++nt) {
    uint32_t qh[8][2], ql[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int d = 16 * kk + 2 * c + 8 * hlf;
        const float2 x = *reinterpret_cast<const float2*>(&qs[8 * nt + g][d]);
        const float h0 = __bfloat162float(__float2bfloat16_rn(x.x));
        const float h1 = __bfloat162float(__float2bfloat16_rn(x.y));
        qh[kk][hlf] = pack_bf16(h0, h1);
        ql[kk][hlf] = pack_bf16(x.x - h0, x.y - h1);
      }
    }
    float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sbase + (kk >> 2) * (kPsRows * 128) + swz128(krow, (kk & 3) * 2 + kchunk), a0, a1, a2, a3);
      mma_bf16(hi, a0, a1, a2, a3, qh[kk][0], qh[kk][1]);
      mma_bf16(lo, a0, a1, a2, a3, ql[kk][0], ql[kk][1]);
    }
    // lane: rows 16 warp + g (+8), tiles 8 nt + 2c and 8 nt + 2c + 1
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t b = chunk0 + 16 * warp + g + 8 * (k >> 1);
      const int tile = t0 + 8 * nt + 2 * c + (k & 1);
      if (b < row_end && tile < t_end) {
        const int64_t n_cand = diag0 + (tile - t0);
        const bool ok = b < n_cand;
        scores[(static_cast<int64_t>(tile) * a.hkv + h) * a.max_blocks + b] = ok ? hi[k] + lo[k] : -INFINITY;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Top-k. grid (Hkv, outer) with outer = batch (decode) or n_tiles (prefill).
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;
// Threads per top-k CTA: a quarter CTA while a unit has at most 4096
// candidates (fewer, cheaper barriers; four CTAs share an SM), else 1024.
inline int topk_threads(int64_t max_blocks) { return max_blocks <= 4096 ? 256 : kTopkThreads; }

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
  int64_t max_blocks;
  PrefillBatch pb;  // prefill: the tiles' sequences
};

constexpr int kCandCap = 8192;  // keys of the threshold bin refined in shared memory

// Finds, among `nbins` counts in shared memory (bin index increasing with the
// key), the bin holding the k-th largest element: *bin and *above (the count
// in higher bins). Each thread owns nbins / blockDim.x consecutive bins.
__device__ inline void find_kth_bin(const int* cnt, int nbins, int k, int* scan_tmp, int* out_bin, int* out_above) {
  const int per = nbins / blockDim.x;
  const int lo = threadIdx.x * per;
  int own = 0;
  for (int j = 0; j < per; ++j) own += cnt[lo + j];
  int total;
  const int incl = block_inclusive_scan(own, scan_tmp, &total);
  int above = total - incl;  // elements in bins above this thread's range
  if (above < k && above + own >= k) {
    for (int j = per - 1; j >= 0; --j) {
      if (above + cnt[lo + j] >= k) {
        *out_bin = lo + j;
        *out_above = above;
        break;
      }
      above += cnt[lo + j];
    }
  }
  __syncthreads();
}

// Histogram of the digit of `bits` bits at `shift` of the keys matching
// (prefix, mask), with warp-aggregated shared-memory atomics (scores of a
// unit crowd into few bins, so lanes with equal digits add once).
__device__ inline void digit_hist(const uint32_t* keys, int n, uint32_t prefix, uint32_t mask, int shift, int bits,
                                  int* cnt) {
  const uint32_t dmask = (1u << bits) - 1u;
  for (int i = threadIdx.x; i < (1 << bits); i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int d = -1;
    if (i < n) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) d = static_cast<int>((key >> shift) & dmask);
    }
    if (d >= 0) atomicAdd(&cnt[d], 1);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, KvView kv, TopkArgs a,
                                                           int32_t* __restrict__ idx_out, int32_t* status) {
  extern __shared__ uint32_t keys[];      // [max_blocks], then kCandCap candidate keys
  __shared__ int cnt[kHistBins];
  __shared__ int scan_tmp[33];
  __shared__ int sel_bin, sel_above, n_cand_keys;

  const int h = blockIdx.x;
  const int outer = blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t unit = static_cast<int64_t>(outer) * a.hkv + h;

  const bool local = (a.force_local & kForceLocal) != 0, sink = (a.force_local & kForceSink) != 0;
  int64_t n64, forced, nb;
  if (!a.prefill) {
    const int64_t len = kv.seq_len(outer, status, kIdTopk);
    nb = (len + kBlock - 1) / kBlock;
    const int64_t nbf = len / kBlock;
    n64 = local ? min(nbf, nb - 1) : nbf;
    forced = (local && nb > 0) ? nb - 1 : -1;
  } else {
    const int s = a.pb.seq_of_tile(outer);
    n64 = a.pb.q_start[s] / kBlock + (outer - a.pb.tile_off[s]);
    nb = n64 + 1;
    forced = local ? n64 : -1;
  }
  if (n64 < 0) n64 = 0;
  // attention sink: block 0 is kept and not scored; the candidates start at 1
  const int skip = (sink && n64 > 0) ? 1 : 0;
  const bool keep0 = sink && nb > 0 && forced != 0;
  const int n = static_cast<int>(n64) - skip;
  const int k = min(a.k_scored, n);
  const float* sc = scores + unit * a.max_blocks + skip;
  int32_t* out = idx_out + unit * a.k_total + (keep0 ? 1 : 0);
  uint32_t* cand = keys + a.max_blocks;

  // eight loads in flight per thread before any store
  for (int base = 0; base < n; base += 8 * static_cast<int>(blockDim.x)) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * blockDim.x + tid;
      v[u] = i < n ? sc[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * blockDim.x + tid;
      if (i < n) keys[i] = float_to_key(v[u]);
    }
  }
  if (tid == 0) n_cand_keys = 0;
  __syncthreads();

  uint32_t thresh = 0;  // the k-th largest key
  int take_equal = 0;   // how many keys equal to thresh are kept (lowest blocks first)
  const bool all = (k >= n);
  if (!all && k > 0) {
    // digit 1: the top 12 bits
    digit_hist(keys, n, 0u, 0u, 32 - kHistBits, kHistBits, cnt);
    find_kth_bin(cnt, kHistBins, k, scan_tmp, &sel_bin, &sel_above);
    uint32_t prefix = static_cast<uint32_t>(sel_bin) << (32 - kHistBits);
    uint32_t mask = 0xFFFFFFFFu << (32 - kHistBits);
    int remaining = k - sel_above;
    const int in_bin = cnt[sel_bin];
    __syncthreads();  // every thread has read in_bin before cnt is reused
    // gather the keys of that bin (few, normally) to refine
    const uint32_t* src = keys;
    int src_n = n;
    if (in_bin <= kCandCap) {
      for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + tid;
        const bool hit = i < n && (keys[i] & mask) == prefix;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        int slot = 0;
        if ((tid & 31) == 0 && m != 0u) slot = atomicAdd(&n_cand_keys, __popc(m));
        slot = __shfl_sync(0xffffffffu, slot, 0);
        if (hit) cand[slot + __popc(m & ((1u << (tid & 31)) - 1u))] = keys[i];
      }
      __syncthreads();
      src = cand;
      src_n = n_cand_keys;
    }
    // digits 2 and 3 (10 bits each)
    for (int shift = 32 - kHistBits - 10; shift >= 0; shift -= 10) {
      digit_hist(src, src_n, prefix, mask, shift, 10, cnt);
      find_kth_bin(cnt, 1024, remaining, scan_tmp, &sel_bin, &sel_above);
      remaining -= sel_above;
      prefix |= static_cast<uint32_t>(sel_bin) << shift;
      mask |= 1023u << shift;
    }
    thresh = prefix;
    take_equal = remaining;
  }

  // Ordered compaction: warp w owns keys [w span, (w + 1) span) and its lanes
  // read consecutive keys (no bank conflicts); ballots order a warp's picks,
  // block scans over the warps' counts order the warps.
  const int lane = tid & 31, nwarps = static_cast<int>(blockDim.x) >> 5;
  const int span = ((n + nwarps - 1) / nwarps + 31) & ~31;
  const int wlo = min(n, (tid >> 5) * span), whi = min(n, wlo + span);
  const unsigned lt = (1u << lane) - 1u;
  int written = 0;
  if (k > 0) {
    int eq_before = 0;  // keys equal to thresh in the warps before this one
    if (!all) {
      int my_eq = 0;
      for (int i = wlo + lane; i < whi; i += 32) my_eq += keys[i] == thresh ? 1 : 0;
      my_eq = __reduce_add_sync(0xffffffffu, my_eq);
      int tot;
      const int v = lane == 0 ? my_eq : 0;
      eq_before = __shfl_sync(0xffffffffu, block_inclusive_scan(v, scan_tmp, &tot) - v, 0);
    }
    // keep: above thresh, or equal to it and among the first take_equal such
    // keys in block order
    auto pass = [&](bool write, int pos) {
      int eq = eq_before, nsel = 0;
      for (int base = wlo; base < whi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < whi ? keys[i] : 0u;
        const bool is_eq = !all && i < whi && key == thresh;
        const unsigned me = __ballot_sync(0xffffffffu, is_eq);
        const bool keep = i < whi && (all || key > thresh || (is_eq && eq + __popc(me & lt) < take_equal));
        const unsigned mk = __ballot_sync(0xffffffffu, keep);
        if (write && keep) out[pos + nsel + __popc(mk & lt)] = static_cast<int32_t>(i + skip);
        nsel += __popc(mk);
        eq += __popc(me);
      }
      return nsel;
    };
    const int nsel = pass(false, 0);
    int tot;
    const int v = lane == 0 ? nsel : 0;
    const int pos = __shfl_sync(0xffffffffu, block_inclusive_scan(v, scan_tmp, &tot) - v, 0);
    pass(true, pos);
    written = tot;
  }
  if (tid == 0) {
    if (keep0) out[-1] = 0;
    int w = written;
    if (forced >= 0) out[w++] = static_cast<int32_t>(forced);
    for (; w + (keep0 ? 1 : 0) < a.k_total; ++w) out[w] = -1;
  }
}

// ---------------------------------------------------------------------------
// Fused decode selection (k_scored <= 64). One CTA handles a chunk of a
// unit's candidate blocks, whose summary rows are one contiguous run for
// either cache layout: bf16 rows are copied into a swizzled shared-memory ring
// by cp.async and scored on the tensor cores, fp32 rows are streamed by a
// producer warp with one bulk copy per stage and scored by a half-warp per
// row; the scores become 64-bit selection keys and the chunk's best are kept
// (a sampled lower bound for bf16, the binned selection otherwise). A unit spread over several chunks posts the chunk
// lists and its last CTA to finish (atomic ticket) selects among them.
// grid (Hkv, batch, n_chunks); chunks past a sequence's candidates exit at
// once and take no ticket.
// ---------------------------------------------------------------------------
constexpr int kSelWarps = 8;
constexpr int kSelThreads = 32 * (kSelWarps + 1);
constexpr int kSelStageRows = 64;
constexpr int kSelStages = 4;
constexpr int kSelStageBytes = kSelStageRows * kHeadDim * 2;  // bf16 rows (fp32 rows use two stages' room)

struct SelDecArgs {
  int hq, hkv;
  int force_local;
  int k_scored;
  int k_total;
  int chunk;        // candidate rows per CTA: 512 * 2^j, <= 4096
  int n_chunks;     // chunks per unit at capacity (grid.x)
  int64_t max_blocks;
  float* scores_out;  // nullable [units, max_blocks]
  uint64_t* cand;     // [units, n_chunks, 64] chunk lists (multi-chunk units)
  int32_t* tickets;   // [units], zero between calls
};

__device__ inline int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Writes the final list of a unit: the blocks of the kk best keys ascending,
// the forced block, then -1 padding. Called by every thread (at least 64);
// top[0..kk) must be visible to all of them. A selected block's position is
// the number of selected blocks below it (the blocks are distinct), counted
// by one thread per block.
__device__ inline void write_selection(const uint64_t* top, int kk, int64_t forced, bool keep0, int k_total,
                                       int32_t* out) {
  const int o = keep0 ? 1 : 0;  // block 0 (attention sink) leads the list
  if (static_cast<int>(threadIdx.x) < kk) {
    // ascending blocks == descending complements (the key's low word)
    const uint32_t me = static_cast<uint32_t>(top[threadIdx.x]);
    int pos = 0;
#pragma unroll 4
    for (int j = 0; j < kk; ++j) pos += static_cast<uint32_t>(top[j]) > me ? 1 : 0;
    out[o + pos] = static_cast<int>(~me);
  }
  for (int i = threadIdx.x; i < k_total; i += blockDim.x) {
    const int j = i - o;
    if (j >= 0 && j < kk) continue;  // a selected block, written above
    out[i] = j < 0 ? 0 : (j == kk && forced >= 0 ? static_cast<int>(forced) : -1);
  }
}

// The k best keys into top[0..k): the binned selection, else (keys crowded
// into one bin) a full sort in lists of 64 using the free ring as scratch.
__device__ inline void choose_top(const uint64_t* keys, int n, int k, uint8_t* ring, uint64_t* top,
                                  SelectScratch& scr, int* count) {
  if (block_select(keys, n, k, top, scr)) return;
  block_topk(keys, n, k, reinterpret_cast<uint64_t*>(ring), top, count);
}

// The k best of n distinct keys through a sampled lower bound: the k-th
// largest of ns sample keys (each the largest of a group of the keys, so
// real keys) bounds the k-th best key from below; the keys at or above it
// (the survivors, a few more than k) are ranked by counting. Returns false,
// the same in every thread, when fewer than k samples are nonzero or more
// than 256 keys survive; the caller then selects otherwise. Every thread of
// the CTA calls this after writing the samples.
__device__ inline bool sampled_top(const uint64_t* keys, int n, int k, const uint64_t* smp, int ns, uint64_t* surv,
                                   uint64_t* top, uint64_t* lb, int* n_surv) {
  const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31;
  if (tid == 0) {
    *lb = 0ull;
    *n_surv = 0;
  }
  __syncthreads();
  if (tid < ns) {
    const uint64_t v = smp[tid];
    int gt = 0, ge = 0;
    for (int j = 0; j < ns; ++j) {
      gt += smp[j] > v ? 1 : 0;
      ge += smp[j] >= v ? 1 : 0;
    }
    if (v != 0ull && gt < k && k <= ge) *lb = v;
  }
  __syncthreads();
  const uint64_t L = *lb;
  if (L == 0ull) return false;
  for (int base = 0; base < n; base += nth) {
    const int i = base + tid;
    const bool hit = i < n && keys[i] >= L;
    const unsigned mk = __ballot_sync(0xffffffffu, hit);
    int slot = 0;
    if (lane == 0 && mk != 0u) slot = atomicAdd(n_surv, __popc(mk));
    slot = __shfl_sync(0xffffffffu, slot, 0);
    const int pos = slot + __popc(mk & ((1u << lane) - 1u));
    if (hit && pos < 256) surv[pos] = keys[i];
  }
  __syncthreads();
  const int m = *n_surv;
  if (m > 256) return false;
  for (int i = tid; i < m; i += nth) {
    const uint64_t x = surv[i];
    int gt = 0;
    for (int j = 0; j < m; ++j) gt += surv[j] > x ? 1 : 0;
    if (gt < k) top[gt] = x;
  }
  __syncthreads();
  return true;
}

// Top-k for k_scored <= 64 and at most 4096 candidates (prefill tiles, and
// decode scores computed apart, as in token-max mode): the scores become
// 64-bit selection keys (score, then lower block first) in shared memory;
// the k best come from a sampled lower bound (the largest key of each of 64
// groups of consecutive keys as the samples), else from the binned
// selection, else (keys crowding one bin) from a radix select of the k-th
// key, which needs no scratch beyond the keys. The list is written as the
// radix top-k writes it. grid (Hkv, outer) with outer = batch (decode) or n_tiles
// (prefill), 256 threads; dynamic shared memory topk64_smem(max_blocks).
constexpr int kTopk64Threads = 256;
constexpr int kTopk64MaxCand = 4096;
static_assert(kTopk64Threads == 4 * 64, "64 sample groups of four threads each");
size_t topk64_smem(int64_t max_blocks) { return static_cast<size_t>(max_blocks) * sizeof(uint64_t); }
__global__ void __launch_bounds__(kTopk64Threads, 8) topk64_kernel(const float* __restrict__ scores, KvView kv, TopkArgs a,
                                                              int32_t* __restrict__ idx_out, int32_t* status) {
  extern __shared__ __align__(16) uint64_t tk[];  // keys [max_blocks]
  __shared__ uint64_t top[64];
  __shared__ SelectScratch scr;
  __shared__ RadixScratch radix;
  __shared__ uint64_t smp[64], lb;
  __shared__ int count, n_surv;
  const int h = blockIdx.x, outer = blockIdx.y;
  const int64_t unit = static_cast<int64_t>(outer) * a.hkv + h;
  const bool local = (a.force_local & kForceLocal) != 0, sink = (a.force_local & kForceSink) != 0;
  pdl_wait();  // the scores come from the previous kernel
  int64_t n64, forced, nb;  // candidates, the kept newest / diagonal block, blocks in view
  if (!a.prefill) {
    const int64_t len = kv.seq_len(outer, status, kIdTopk);
    nb = (len + kBlock - 1) / kBlock;
    const int64_t nbf = len / kBlock;
    n64 = local ? min(nbf, nb - 1) : nbf;
    forced = (local && nb > 0) ? nb - 1 : -1;
  } else {
    const int seq = a.pb.seq_of_tile(outer);
    n64 = a.pb.q_start[seq] / kBlock + (outer - a.pb.tile_off[seq]);  // blocks before the diagonal
    nb = n64 + 1;
    forced = local ? n64 : -1;
  }
  if (n64 < 0) n64 = 0;
  const int skip = (sink && n64 > 0) ? 1 : 0;  // attention sink: block 0 kept, not scored
  const bool keep0 = sink && nb > 0 && forced != 0;
  const int n = static_cast<int>(n64) - skip;
  const int k = min(a.k_scored, n);
  const float* sc = scores + unit * a.max_blocks;
  // the score loads eight at a time in flight, then their keys
  for (int base = 0; base < n; base += 8 * kTopk64Threads) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + threadIdx.x + u * kTopk64Threads;
      v[u] = i < n ? sc[i + skip] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + threadIdx.x + u * kTopk64Threads;
      if (i < n) tk[i] = sel_key(v[u], i + skip);
    }
  }
  __syncthreads();
  {
    // sample g: the largest key of keys [g G, (g + 1) G), four threads a group
    const int G = (n + 63) / 64, g = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int end = min(n, (g + 1) * G);
    uint64_t m = 0ull;
    for (int i = g * G + part; i < end; i += 4) m = tk[i] > m ? tk[i] : m;
    uint64_t o = shfl_xor_u64(m, 1);
    m = o > m ? o : m;
    o = shfl_xor_u64(m, 2);
    m = o > m ? o : m;
    if (part == 0) smp[g] = m;
  }
  if (k > 0 && !sampled_top(tk, n, k, smp, 64, scr.cand, top, &lb, &n_surv) && !block_select(tk, n, k, top, scr))
    block_compact_ge(tk, n, block_kth_largest(tk, n, k, radix), top, 64, &count);  // exactly the k best
  pdl_trigger();  // the attention kernel may start its set-up
  write_selection(top, max(k, 0), forced, keep0, a.k_total, idx_out + unit * a.k_total);
}

template <typename T>
__global__ void __launch_bounds__(kSelThreads, 2) select_decode_kernel(const T* __restrict__ q,
                                                                   const T* __restrict__ pooled, KvView kv,
                                                                   SelDecArgs a, int32_t* __restrict__ idx_out,
                                                                   int32_t* status) {
  constexpr int kRowBytes = SelRow<T>::kBytes;
  constexpr int kStageRows = kSelStageBytes / kRowBytes;  // 64 (bf16) or 32 (fp32) rows per stage
  extern __shared__ __align__(128) uint8_t sel_raw[];
  uint8_t* ring = sel_raw;                                                   // kSelStages x 16 KB
  uint64_t* keys = reinterpret_cast<uint64_t*>(sel_raw + kSelStages * kSelStageBytes);  // [max(chunk, 2048)]
  __shared__ uint64_t full[kSelStages], empty[kSelStages];
  __shared__ uint64_t top[64];
  __shared__ SelectScratch scr;
  __shared__ int count, is_last;

  // chunk pieces are dispatched deepest first (grid z descending): the long
  // units' full pieces start first and the small ones fill in behind them
  const int c = static_cast<int>(gridDim.z) - 1 - static_cast<int>(blockIdx.z);
  const int h = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = static_cast<int64_t>(s) * a.hkv + h;
  const int grp = a.hq / a.hkv;
  pdl_wait();  // inputs and the workspace may come from the previous kernel

  const int64_t len = kv.seq_len(s, status, kIdScore);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  const int64_t nbf = len / kBlock;
  const bool local = (a.force_local & kForceLocal) != 0, sink = (a.force_local & kForceSink) != 0;
  int64_t n_cand = local ? min(nbf, nb - 1) : nbf;
  if (n_cand < 0) n_cand = 0;
  const int64_t forced = (local && nb > 0) ? nb - 1 : -1;
  const int skip = (sink && n_cand > 0) ? 1 : 0;     // attention sink: block 0 kept, not scored
  const bool keep0 = sink && nb > 0 && forced != 0;
  const int my_chunks = n_cand > 0 ? static_cast<int>((n_cand + a.chunk - 1) / a.chunk) : 1;
  if (c >= my_chunks) return;  // past this sequence's candidates
  // piece 0 is the partial one: rows [0, p); piece c >= 1 is rows
  // [p + (c - 1) chunk, p + c chunk), a full chunk
  const int64_t p0 = n_cand - static_cast<int64_t>(my_chunks - 1) * a.chunk;
  const int64_t r0 = c == 0 ? 0 : p0 + static_cast<int64_t>(c - 1) * a.chunk;
  const int rows = static_cast<int>(max(static_cast<int64_t>(0), c == 0 ? p0 : static_cast<int64_t>(a.chunk)));
  const int n_stages = (rows + kStageRows - 1) / kStageRows;

  if (tid == 0) {
    for (int i = 0; i < kSelStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kSelWarps);
    }
    fence_mbar_init();
  }
  // bf16: the group's query rows are loaded now and summed after the set-up
  // barrier
  float xq[kMaxGroupHeads];
  if constexpr (sizeof(T) == 2) {
    if (tid < kHeadDim) {
      const T* qg = q + (static_cast<int64_t>(s) * a.hq + h * grp) * kHeadDim + tid;
#pragma unroll
      for (int g = 0; g < kMaxGroupHeads; ++g) xq[g] = g < grp ? __bfloat162float(qg[g * kHeadDim]) : 0.f;
    }
  }
  __syncthreads();

  auto emit = [&](int i, float part, bool ok) -> uint64_t {  // row i of the chunk
    const int64_t b = r0 + i;
    ok = ok && !(skip && b == 0);
    const uint64_t key = ok ? sel_key(part, static_cast<int>(b)) : 0ull;
    keys[i] = key;
    if (a.scores_out != nullptr) a.scores_out[unit * a.max_blocks + b] = ok ? part : -INFINITY;
    return key;
  };
  // bf16: each scoring lane's largest key of its even and of its odd stages,
  // 64 samples for the sampled bound of the chunk's top-k
  __shared__ uint64_t smp[64];
  uint64_t smax0 = 0ull, smax1 = 0ull;
  if constexpr (sizeof(T) == 2) {
    // bf16: every compute thread gathers 16-byte pieces of the stage's 64
    // summary rows (one contiguous run per unit, either cache layout) with cp.async into
    // a 4-stage ring, 128-byte swizzled as [64-dim half][row][128 B]; warps
    // 0-3 score 16 rows each on the tensor cores with the index query split
    // into a bf16 head and remainder (as in the fused step).
    constexpr int kRows = kSelStageBytes / (kHeadDim * 2);  // 64 rows per stage
    const int64_t contig0 = (static_cast<int64_t>(s) * a.hkv + h) * a.max_blocks + r0;
    auto issue = [&](int st) {
      if (st < n_stages && warp < kSelWarps) {
        uint8_t* stage = ring + (st % kSelStages) * kSelStageBytes;
        const int base = st * kRows;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = tid + 32 * kSelWarps * u;  // 1024 pieces: row j / 16, piece j % 16
          const int row = j >> 4, pc = j & 15;
          const int i = base + row;
          if (i >= rows) continue;
          cp_async16(stage + (pc >> 3) * (kRows * 128) + row * 128 + (((pc & 7) ^ (row & 7)) << 4),
                     pooled + (contig0 + i) * kHeadDim + 8 * pc);
        }
      }
      cp_async_commit();
    };
    // the first stages are in flight before the index query is summed (its
    // rows were loaded before the set-up barrier)
    for (int st = 0; st < kSelStages - 1; ++st) issue(st);
    __shared__ float qsum[kHeadDim];
    if (tid < kHeadDim) {
      float acc = 0.f;
#pragma unroll
      for (int g = 0; g < kMaxGroupHeads; ++g) acc += xq[g];
      qsum[tid] = acc;
    }
    __syncthreads();
    const int g = lane >> 2, c = lane & 3;
    uint32_t qb[8][2];
#pragma unroll
    for (int kk2 = 0; kk2 < 8; ++kk2) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int d = 16 * kk2 + 2 * c + 8 * hlf;
        float x0 = qsum[d], x1 = qsum[d + 1];
        if (g == 1) {
          x0 -= __bfloat162float(__float2bfloat16_rn(x0));
          x1 -= __bfloat162float(__float2bfloat16_rn(x1));
        }
        qb[kk2][hlf] = g < 2 ? pack_bf16(x0, x1) : 0u;
      }
    }
    const int krow = 16 * (warp & 3) + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kchunk = lane >> 4;
    for (int st = 0; st < n_stages; ++st) {
      cp_async_wait<kSelStages - 2>();
      __syncthreads();  // stage st has landed for every thread; stage st - 1 is consumed
      issue(st + kSelStages - 1);
      if (warp < 4) {
        const uint32_t sbase = smem_u32(ring + (st % kSelStages) * kSelStageBytes);
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk2 = 0; kk2 < 8; ++kk2) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(sbase + (kk2 >> 2) * (kRows * 128) + swz128(krow, (kk2 & 3) * 2 + kchunk), a0, a1, a2, a3);
          mma_bf16(sacc, a0, a1, a2, a3, qb[kk2][0], qb[kk2][1]);
        }
        if (c == 0) {
          const int base = st * kRows;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int i = base + 16 * warp + g + 8 * hh;
            if (i < rows) {
              const uint64_t kx = emit(i, sacc[2 * hh] + sacc[2 * hh + 1], true);
              if (st & 1) smax1 = kx > smax1 ? kx : smax1;
              else smax0 = kx > smax0 ? kx : smax0;
            }
          }
        }
      }
    }
    cp_async_wait<0>();
  } else {
  const int e = tid & 15, hw = tid >> 4;  // scorers: 16 half-warps, lane e owns dims [8e, 8e+8)
  float qi[8];
  if (warp < kSelWarps) {
#pragma unroll
    for (int i = 0; i < 8; ++i) qi[i] = 0.f;
    for (int g = 0; g < grp; ++g) {
      float x[8];
      load8<T>(q + (static_cast<int64_t>(s) * a.hq + h * grp + g) * kHeadDim + 8 * e, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) qi[i] += x[i];
    }
  }
  {
    if (warp == kSelWarps) {
      // ---------------- producer: one bulk copy per stage ----------------
      if (lane == 0) {
        int issued = 0;
        for (int st = 0; st < n_stages; ++st) {
          const int slot = st % kSelStages;
          if (st >= kSelStages && !mbar_wait(&empty[slot], ((st / kSelStages) - 1) & 1, status, kIdScore)) break;
          const int base = st * kStageRows;
          const int n = min(kStageRows, rows - base);
          const T* src = pooled + ((static_cast<int64_t>(s) * a.hkv + h) * a.max_blocks + r0 + base) * kHeadDim;
          mbar_arrive_expect_tx(&full[slot], n * kRowBytes);
          bulk_load(ring + slot * kSelStageBytes, src, n * kRowBytes, &full[slot]);
          issued = st + 1;
        }
        mbar_drain(full, kSelStages, issued, status, kIdScore);
      }
    } else {
      // ---------------- scorers ----------------
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % kSelStages;
        if (!mbar_wait_warp(&full[slot], (st / kSelStages) & 1, status, kIdScore)) break;
        const uint8_t* stage = ring + slot * kSelStageBytes;
        const int base = st * kStageRows;
        const int n = min(kStageRows, rows - base);
#pragma unroll
        for (int rr = 0; rr < kStageRows / 16; ++rr) {
          const int i = rr * 16 + hw;  // row within the stage
          float part = i < n ? SelRow<T>::dot(stage + i * kRowBytes, e, qi) : 0.f;
          part += __shfl_xor_sync(0xffffffffu, part, 8);
          part += __shfl_xor_sync(0xffffffffu, part, 4);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          if (e == 0 && i < n) emit(base + i, part, true);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
    }
  }
  }  // fp32 rows
  __syncthreads();
  pdl_trigger();  // the attention kernel may start its set-up
  const int kk = static_cast<int>(n_cand - skip < a.k_scored ? n_cand - skip : static_cast<int64_t>(a.k_scored));
  int32_t* out = idx_out + unit * a.k_total;
  const int kk_local = min(kk, rows - (c == 0 ? skip : 0));
  if (kk_local > 0) {
    bool done = false;
    if constexpr (sizeof(T) == 2) {
      __shared__ uint64_t s_lb;
      __shared__ int s_nsurv;
      if (warp < 4 && (lane & 3) == 0) {
        smp[2 * (8 * warp + (lane >> 2))] = smax0;
        smp[2 * (8 * warp + (lane >> 2)) + 1] = smax1;
      }
      done = sampled_top(keys, rows, kk_local, smp, 64, reinterpret_cast<uint64_t*>(ring), top, &s_lb, &s_nsurv);
    }
    if (!done) choose_top(keys, rows, kk_local, ring, top, scr, &count);
  }
  if (my_chunks == 1) {
    write_selection(top, kk, forced, keep0, a.k_total, out);
    return;
  }
  // post this chunk's list; the unit's last CTA selects among them
  uint64_t* mine = a.cand + (unit * a.n_chunks + c) * 64;
  if (tid < 64) mine[tid] = tid < kk_local ? top[tid] : 0ull;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&a.tickets[unit], 1) == my_chunks - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const uint64_t* all = a.cand + unit * a.n_chunks * 64;
  const int n_all = my_chunks * 64;
  for (int i = tid; i < n_all; i += blockDim.x) keys[i] = __ldcg(all + i);
  __syncthreads();
  if (kk > 0) choose_top(keys, n_all, kk, ring, top, scr, &count);
  write_selection(top, kk, forced, keep0, a.k_total, out);
  if (tid == 0) a.tickets[unit] = 0;  // ready for the next call
}

// Chunk size for the decode selection kernel: 2048 candidate rows (fewer,
// longer CTAs amortise their fixed costs: index query, top-k, list merge),
// halved down to 512 while the grid would hold fewer than two CTAs per SM,
// then doubled while a unit would need more than 32 chunks (the last chunk of
// a unit merges at most 32 lists of 64). Chunks past a short sequence's
// candidates exit at once, so a ragged batch sized by its longest sequence
// costs little.
void select_decode_shape(int64_t max_blocks, int64_t units, int num_sms, int* chunk, int* n_chunks) {
  int c = 2048;
  while (c > 512 && units * ((max_blocks + c - 1) / c) < 2LL * num_sms) c >>= 1;
  while (c < 4096 && (max_blocks + c - 1) / c > 32) c <<= 1;
  *chunk = c;
  *n_chunks = static_cast<int>((max_blocks + c - 1) / c);
  if (*n_chunks < 1) *n_chunks = 1;
}

size_t select_decode_smem(int chunk) {
  const int n = chunk > 2048 ? chunk : 2048;
  return static_cast<size_t>(kSelStages) * kSelStageBytes + static_cast<size_t>(n) * sizeof(uint64_t);
}

size_t select_decode_cand_bytes(int64_t units, int n_chunks) {
  return static_cast<size_t>(units) * n_chunks * 64 * sizeof(uint64_t);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
// The top-k over scores in `scores`: the key-based kernel for k <= 64 of at
// most 4096 candidates, else the radix select. grid (Hkv, outer).
static cudaError_t launch_topk(const float* scores, const KvView& kv, const TopkArgs& ta, int outer,
                               int32_t* idx_out, int32_t* status, cudaStream_t stream) {
  if (ta.k_scored <= 64 && ta.max_blocks <= kTopk64MaxCand) {
    // programmatic dependent launch: the CTAs may be placed while the score
    // kernel drains; they wait for its results before reading anything
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(kv.hkv, outer, 1);
    lc.blockDim = dim3(kTopk64Threads, 1, 1);
    lc.dynamicSmemBytes = topk64_smem(ta.max_blocks);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, topk64_kernel, scores, kv, ta, idx_out, status);
  }
  const size_t smem = static_cast<size_t>(ta.max_blocks + kCandCap) * sizeof(uint32_t);
  topk_kernel<<<dim3(kv.hkv, outer), topk_threads(ta.max_blocks), smem, stream>>>(scores, kv, ta, idx_out, status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_select(const T* q, int hq, const PrefillBatch* pb, const T* pooled, const KvView& kv, int batch,
                          const msa_select_cfg& cfg, int32_t* idx_out, int k_total, float* scores, float* qidx_ws,
                          const FusedSelect* fused, int32_t* status, cudaStream_t stream) {
  const int prefill = cfg.q_tile == kBlock;
  const int64_t max_blocks = kv.max_blocks();
  ScoreArgs sa{hq, kv.hkv, prefill, cfg.force_local, prefill ? pb->q_start[0] : 0, 0, max_blocks};
  const unsigned chunks = static_cast<unsigned>((max_blocks + kScoreChunk - 1) / kScoreChunk);
  int outer;
  if (!prefill && cfg.k_scored <= 64 && fused != nullptr) {
    SelDecArgs da;
    da.hq = hq;
    da.hkv = kv.hkv;
    da.force_local = cfg.force_local;
    da.k_scored = cfg.k_scored;
    da.k_total = k_total;
    select_decode_shape(max_blocks, static_cast<int64_t>(batch) * kv.hkv, fused->num_sms, &da.chunk, &da.n_chunks);
    da.max_blocks = max_blocks;
    da.scores_out = fused->scores_out;
    da.cand = fused->cand;
    da.tickets = fused->tickets;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(kv.hkv, batch, da.n_chunks);
    lc.blockDim = dim3(kSelThreads, 1, 1);
    lc.dynamicSmemBytes = select_decode_smem(da.chunk);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, select_decode_kernel<T>, q, pooled, kv, da, idx_out, status);
  }
  if (!prefill) {
    outer = batch;
    score_kernel<T, 1><<<dim3(chunks, kv.hkv, batch), kScoreThreads, 0, stream>>>(q, nullptr, pooled, kv, sa,
                                                                                  scores, status);
  } else {
    const int n_tiles = pb->total_tiles();
    outer = n_tiles;
    sa.n_tiles = n_tiles;
    if constexpr (sizeof(T) == 2) {
      const size_t smem = kQidxSmemMax;
      qidx_prefill_bf16_kernel<<<dim3(kv.hkv, n_tiles), kQidxThreads, smem, stream>>>(q, hq, kv.hkv, *pb, qidx_ws);
    } else {
      qidx_prefill_kernel<T><<<dim3(kv.hkv, n_tiles), 256, 0, stream>>>(q, hq, kv.hkv, *pb, qidx_ws);
    }
    constexpr int kT = 8;
    // only the chunks below the last tile's diagonal hold candidates
    int64_t last = 0;
    for (int s = 0; s < pb->n_seqs; ++s)
      last = max(last, pb->q_start[s] / kBlock + (pb->tile_off[s + 1] - pb->tile_off[s]));
    if constexpr (sizeof(T) == 2) {
      const unsigned pchunks = static_cast<unsigned>((min(last, max_blocks) + kPsRows - 1) / kPsRows);
      score_prefill_mma_kernel<<<dim3(pchunks, kv.hkv, pb->grp_off[pb->n_seqs]), 256, 0, stream>>>(
          qidx_ws, pooled, kv, sa, *pb, scores, status);
    } else {  // fp32 prefill selection: one sequence
      const unsigned pchunks = static_cast<unsigned>((min(last, max_blocks) + kScoreChunk - 1) / kScoreChunk);
      score_kernel<T, kT><<<dim3(pchunks, kv.hkv, (n_tiles + kT - 1) / kT), kScoreThreads, 0, stream>>>(
          q, qidx_ws, pooled, kv, sa, scores, status);
    }
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  TopkArgs ta{kv.hkv, prefill, cfg.force_local, cfg.k_scored, k_total, max_blocks, {}};
  if (prefill) ta.pb = *pb;
  return launch_topk(scores, kv, ta, outer, idx_out, status, stream);
}

// Top-k over decode scores already in `scores` ([batch, hkv, max_blocks]).
cudaError_t launch_topk_scores(const float* scores, const KvView& kv, int batch, const msa_select_cfg& cfg,
                               int32_t* idx_out, int k_total, int32_t* status, cudaStream_t stream) {
  TopkArgs ta{kv.hkv, 0, cfg.force_local, cfg.k_scored, k_total, kv.max_blocks(), {}};
  return launch_topk(scores, kv, ta, batch, idx_out, status, stream);
}

// Token-max selection of prefill tiles (bf16): the tiles' index queries, the
// token-level block maxima against the shared index-key head, then the top-k.
cudaError_t launch_select_token_max_prefill(const CUtensorMap& tmi, const __nv_bfloat16* q, int hq,
                                            const PrefillBatch& pb, const KvView& kv, const msa_select_cfg& cfg,
                                            int32_t* idx_out, int k_total, float* scores, float* qidx_ws,
                                            int32_t* status, cudaStream_t stream) {
  const int n_tiles = pb.total_tiles();
  const size_t smem = kQidxSmemMax;
  qidx_prefill_bf16_kernel<<<dim3(kv.hkv, n_tiles), kQidxThreads, smem, stream>>>(q, hq, kv.hkv, pb, qidx_ws);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if ((err = launch_token_max_prefill_scores(tmi, kv, pb, qidx_ws, scores, status, stream)) != cudaSuccess) return err;
  TopkArgs ta{kv.hkv, 1, cfg.force_local, cfg.k_scored, k_total, kv.max_blocks(), pb};
  return launch_topk(scores, kv, ta, n_tiles, idx_out, status, stream);
}

cudaError_t set_select_decode_smem(size_t bytes) {
  // the decode step's kernels all ask for the largest shared-memory carve-out,
  // so consecutive launches need no L1/shared reconfiguration
  const void* fns[2] = {reinterpret_cast<const void*>(select_decode_kernel<__nv_bfloat16>),
                        reinterpret_cast<const void*>(select_decode_kernel<float>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t set_qidx_smem() {
  cudaError_t e = cudaFuncSetAttribute(qidx_prefill_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kQidxSmemMax));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topk64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(topk64_smem(kTopk64MaxCand)));
}

cudaError_t set_topk_smem(size_t bytes) {
  return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template cudaError_t launch_select<__nv_bfloat16>(const __nv_bfloat16*, int, const PrefillBatch*,
                                                  const __nv_bfloat16*, const KvView&, int, const msa_select_cfg&,
                                                  int32_t*, int, float*, float*, const FusedSelect*, int32_t*,
                                                  cudaStream_t);
template cudaError_t launch_select<float>(const float*, int, const PrefillBatch*, const float*, const KvView&, int,
                                          const msa_select_cfg&, int32_t*, int, float*, float*, const FusedSelect*,
                                          int32_t*, cudaStream_t);

bool make_prefill_batch(int n_seqs, const int64_t* q_starts, const int32_t* q_counts, PrefillBatch* b) {
  if (n_seqs < 1 || n_seqs > kMaxPrefillSeqs || q_starts == nullptr || q_counts == nullptr) return false;
  *b = PrefillBatch{};
  b->n_seqs = n_seqs;
  int32_t off = 0, tiles = 0, groups = 0;
  for (int s = 0; s < n_seqs; ++s) {
    if (q_counts[s] < 0 || q_starts[s] < 0) return false;
    b->q_start[s] = q_starts[s];
    b->q_off[s] = off;
    b->q_cnt[s] = q_counts[s];
    b->tile_off[s] = tiles;
    b->grp_off[s] = groups;
    const int32_t t = chunk_tiles(q_starts[s], q_counts[s]);
    off += q_counts[s];
    tiles += t;
    groups += (t + kPsTiles - 1) / kPsTiles;
  }
  b->tile_off[n_seqs] = tiles;
  b->grp_off[n_seqs] = groups;
  return true;
}

}  // namespace msa
