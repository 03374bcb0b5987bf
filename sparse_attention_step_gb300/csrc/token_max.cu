// Step 1 as the guide draws it ("MiniMax goes sparse", §1 Step 1): token-level
// index scores q_idx . K_idx[t] against a single index-key head shared by every
// GQA group of the layer, then a max pool over the 64 tokens of each block.
//
// One CTA scores a chunk of a sequence's candidate blocks for all of its KV
// heads at once (the index keys are shared, so each is read once per step):
// a producer warp streams each 64-token block of index keys with two 2-D TMA
// boxes (128-byte swizzle) into a 4-stage ring; four warps take 16 tokens each
// and compute S[token, group] = K_idx q_idx^T with mma.sync, the fp32 index
// queries of up to 8 groups split into a bf16 head (one n-tile) and a bf16
// remainder (a second n-tile), then reduce the max over their tokens. The
// block maxima go to the score buffer that the top-k kernel reads.
#include <float.h>

#include "kernels.cuh"

namespace msa {

namespace {

constexpr int kTmWarps = 4;
constexpr int kTmThreads = 32 * (kTmWarps + 1);
constexpr int kTmStages = 4;
constexpr int kTmStage = kBlock * kHeadDim * 2;  // 16 KB: one block of index keys
constexpr int kTmMaxChunk = 64;                  // candidate blocks per CTA, at most
constexpr int kTmCtasPerSm = 3;                  // resident CTAs per SM (65 KB of shared memory each)
constexpr int kTmMaxHeads = 8;

}  // namespace

struct TokenMaxArgs {
  const __nv_bfloat16* q;  // [batch, hq, 128]
  int hq, hkv, grp;
  int force_local;
  int chunk;  // candidate blocks per CTA, <= kTmMaxChunk
  int64_t max_blocks;
  float* scores;  // [batch, hkv, max_blocks]
  int32_t* status;
};

// grid (chunks, batch)
__global__ void __launch_bounds__(kTmThreads) token_max_score_kernel(const __grid_constant__ CUtensorMap tmi,
                                                                     KvView kv, TokenMaxArgs a) {
  extern __shared__ __align__(1024) uint8_t tm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kTmStages], empty[kTmStages];
  __shared__ float qsum[kTmMaxHeads][kHeadDim];
  __shared__ int32_t rowid[kTmMaxChunk];                      // first index-key row of each block, -1 = bad page
  __shared__ float part[kTmMaxChunk][kTmWarps][kTmMaxHeads];  // per-warp block maxima

  const int s = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  const int64_t len = kv.seq_len(s, a.status, kIdScore);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  const int64_t nbf = len / kBlock;
  int64_t n_cand = (a.force_local & kForceLocal) ? min(nbf, nb - 1) : nbf;
  if (n_cand < 0) n_cand = 0;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * a.chunk;
  if (b0 >= n_cand) return;
  const int nblk = static_cast<int>(min(static_cast<int64_t>(a.chunk), n_cand - b0));

  if (tid == 0) {
    for (int i = 0; i < kTmStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kTmWarps);
    }
    fence_mbar_init();
  }
  if (tid < kTmMaxChunk) {
    int32_t r = -1;
    if (tid < nblk) {
      const int64_t b = b0 + tid;
      if (kv.layout == MSA_KV_CONTIGUOUS) {
        r = static_cast<int32_t>(static_cast<int64_t>(s) * kv.max_tokens + b * kBlock);
      } else {
        const int32_t p = kv.page(s, b, a.status, kIdScore);
        r = p < 0 ? -1 : p * kBlock;
      }
    }
    rowid[tid] = r;
  }
  for (int i = tid; i < kTmMaxHeads * kHeadDim; i += blockDim.x) {
    const int h = i / kHeadDim, d = i % kHeadDim;
    float acc = 0.f;
    if (h < a.hkv) {
      const __nv_bfloat16* qg = a.q + (static_cast<int64_t>(s) * a.hq + h * a.grp) * kHeadDim + d;
      float x[kMaxGroupHeads];
#pragma unroll
      for (int g = 0; g < kMaxGroupHeads; ++g) x[g] = g < a.grp ? __bfloat162float(qg[g * kHeadDim]) : 0.f;
#pragma unroll
      for (int g = 0; g < kMaxGroupHeads; ++g) acc += x[g];
    }
    qsum[h][d] = acc;
  }
  __syncthreads();

  if (warp == kTmWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tmi);
      for (int j = 0; j < nblk; ++j) {
        const int slot = j % kTmStages;
        if (j >= kTmStages && !mbar_wait(&empty[slot], ((j / kTmStages) - 1) & 1, a.status, kIdScore)) break;
        const int32_t y = rowid[j] < 0 ? 0 : rowid[j];
        uint8_t* dst = ring + slot * kTmStage;
        mbar_arrive_expect_tx(&full[slot], kTmStage);
        tma_load_2d(dst, &tmi, 0, y, &full[slot]);
        tma_load_2d(dst + kTmStage / 2, &tmi, 64, y, &full[slot]);
      }
    }
  } else {
    const int g = lane >> 2, c = lane & 3;
    // B operands: column n = group g; n-tile 0 the bf16 head, n-tile 1 the remainder
    uint32_t qh[8][2], ql[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int d = 16 * kk + 2 * c + 8 * hlf;
        const float x0 = qsum[g][d], x1 = qsum[g][d + 1];
        const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
        const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
        qh[kk][hlf] = pack_bf16(h0, h1);
        ql[kk][hlf] = pack_bf16(x0 - h0, x1 - h1);
      }
    }
    const int krow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kchunk = lane >> 4;
    for (int j = 0; j < nblk; ++j) {
      const int slot = j % kTmStages;
      if (!mbar_wait_warp(&full[slot], (j / kTmStages) & 1, a.status, kIdScore)) break;
      const uint32_t sbase = smem_u32(ring + slot * kTmStage);
      float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sbase + (kk >> 2) * (kTmStage / 2) + swz128(krow, (kk & 3) * 2 + kchunk), a0, a1, a2, a3);
        mma_bf16(hi, a0, a1, a2, a3, qh[kk][0], qh[kk][1]);
        mma_bf16(lo, a0, a1, a2, a3, ql[kk][0], ql[kk][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      // tokens g and g + 8 of this warp's 16, groups 2c and 2c + 1
      float m0 = fmaxf(hi[0] + lo[0], hi[2] + lo[2]);
      float m1 = fmaxf(hi[1] + lo[1], hi[3] + lo[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
      }
      if (g == 0) {
        part[j][warp][2 * c] = m0;
        part[j][warp][2 * c + 1] = m1;
      }
    }
  }
  pdl_trigger();
  __syncthreads();
  for (int i = tid; i < nblk * a.hkv; i += blockDim.x) {
    const int j = i / a.hkv, h = i % a.hkv;
    float m = fmaxf(fmaxf(part[j][0][h], part[j][1][h]), fmaxf(part[j][2][h], part[j][3][h]));
    if (rowid[j] < 0) m = -INFINITY;  // bad page: never selected
    a.scores[(static_cast<int64_t>(s) * a.hkv + h) * a.max_blocks + b0 + j] = m;
  }
}

// ---------------------------------------------------------------------------
// Prefill tiles: the same token-level max-pooled score, for the 64-token query
// tiles of a chunk batch. A CTA takes a chunk of index-key blocks of one
// sequence and a group of up to 8 of its tiles, for every KV head: per block
// and head, S[token, tile] = K_idx q_idx(tile, head)^T on mma.sync (the tiles
// are the 8 columns; the fp32 index queries split into a bf16 head and a bf16
// remainder, as above), and the max over the block's 64 tokens (four warps of
// 16 tokens, combined with shared-memory atomics on order-preserving keys).
// The index queries come from the workspace (the prefill index-query kernel).
// grid (block chunks, tile groups).
// ---------------------------------------------------------------------------
namespace {
constexpr int kTpTiles = 8;   // tiles per group (the MMA's N)
constexpr int kTpChunk = 32;  // index-key blocks per CTA (two CTAs fit an SM)
}  // namespace

struct TokenMaxPrefillArgs {
  const float* qidx;  // [tiles, hkv, 128] fp32
  int hkv;
  int64_t max_blocks;
  float* scores;  // [tiles, hkv, max_blocks]
  int32_t* status;
};

__global__ void __launch_bounds__(kTmThreads) token_max_prefill_kernel(const __grid_constant__ CUtensorMap tmi,
                                                                       KvView kv, TokenMaxPrefillArgs a,
                                                                       const PrefillBatch pb) {
  extern __shared__ __align__(1024) uint8_t tp_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tp_raw) + 1023) & ~uintptr_t(1023));
  // B fragments [head][kk][hlf][head / remainder][lane] and the block maxima as keys [block][head][tile]
  uint32_t* qb = reinterpret_cast<uint32_t*>(ring + kTmStages * kTmStage);
  uint32_t* part = qb + kTmMaxHeads * 8 * 2 * 2 * 32;
  __shared__ uint64_t full[kTmStages], empty[kTmStages];
  __shared__ int32_t rowid[kTpChunk];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = pb.seq_of_group(blockIdx.y);
  const int j0 = (blockIdx.y - pb.grp_off[seq]) * kTpTiles;      // first tile of the group within its sequence
  const int t0 = pb.tile_off[seq] + j0;                          // its global tile
  const int t_end = min(t0 + kTpTiles, pb.tile_off[seq + 1]);
  const int64_t diag0 = pb.q_start[seq] / kBlock + j0;           // candidates of tile t0 + t: blocks < diag0 + t
  const int64_t n_max = diag0 + (t_end - t0) - 1;                // the group's most candidates
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kTpChunk;
  if (b0 >= n_max) return;
  const int nblk = static_cast<int>(min(static_cast<int64_t>(kTpChunk), n_max - b0));
  pdl_wait();

  if (tid == 0) {
    for (int i = 0; i < kTmStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kTmWarps);
    }
    fence_mbar_init();
  }
  if (tid < kTpChunk) {
    int32_t r = -1;
    if (tid < nblk) {
      const int64_t b = b0 + tid;
      if (kv.layout == MSA_KV_CONTIGUOUS) {
        r = static_cast<int32_t>(static_cast<int64_t>(seq) * kv.max_tokens + b * kBlock);
      } else {
        const int32_t p = kv.page(seq, b, a.status, kIdScore);
        r = p < 0 ? -1 : p * kBlock;
      }
    }
    rowid[tid] = r;
  }
  for (int i = tid; i < kTmMaxHeads * 8 * 2 * 32; i += blockDim.x) {
    const int ln = i & 31, hlf = (i >> 5) & 1, kk = (i >> 6) & 7, h = i >> 9;
    const int g = ln >> 2, c = ln & 3;
    const int d = 16 * kk + 2 * c + 8 * hlf;
    float x0 = 0.f, x1 = 0.f;
    if (h < a.hkv && t0 + g < t_end) {
      const float* qi = a.qidx + (static_cast<int64_t>(t0 + g) * a.hkv + h) * kHeadDim;
      x0 = qi[d];
      x1 = qi[d + 1];
    }
    const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
    const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
    const int at = (((h * 8 + kk) * 2 + hlf) * 2) * 32 + ln;
    qb[at] = pack_bf16(h0, h1);
    qb[at + 32] = pack_bf16(x0 - h0, x1 - h1);
  }
  const uint32_t neg_inf = float_to_key(-INFINITY);
  for (int i = tid; i < kTpChunk * kTmMaxHeads * kTpTiles; i += blockDim.x) part[i] = neg_inf;
  __syncthreads();

  if (warp == kTmWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tmi);
      for (int j = 0; j < nblk; ++j) {
        const int slot = j % kTmStages;
        if (j >= kTmStages && !mbar_wait(&empty[slot], ((j / kTmStages) - 1) & 1, a.status, kIdScore)) break;
        const int32_t y = rowid[j] < 0 ? 0 : rowid[j];
        uint8_t* dst = ring + slot * kTmStage;
        mbar_arrive_expect_tx(&full[slot], kTmStage);
        tma_load_2d(dst, &tmi, 0, y, &full[slot]);
        tma_load_2d(dst + kTmStage / 2, &tmi, 64, y, &full[slot]);
      }
    }
  } else {
    const int c = lane & 3;
    const int krow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kchunk = lane >> 4;
    for (int j = 0; j < nblk; ++j) {
      const int slot = j % kTmStages;
      if (!mbar_wait_warp(&full[slot], (j / kTmStages) & 1, a.status, kIdScore)) break;
      const uint32_t sbase = smem_u32(ring + slot * kTmStage);
      uint32_t af[8][4];  // this warp's 16 tokens of the block, all 128 dims
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        ldsm_x4(sbase + (kk >> 2) * (kTmStage / 2) + swz128(krow, (kk & 3) * 2 + kchunk), af[kk][0], af[kk][1],
                af[kk][2], af[kk][3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      // every head's products at once (16 independent accumulator chains per
      // k-step), so the tensor pipe, not the chain latency, sets the pace
      float hi[kTmMaxHeads][4], lo[kTmMaxHeads][4];
#pragma unroll
      for (int h = 0; h < kTmMaxHeads; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) hi[h][e] = lo[h][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int h = 0; h < kTmMaxHeads; ++h) {
          if (h < a.hkv) {
            const uint32_t* qh = qb + h * (8 * 2 * 2 * 32) + lane;
            mma_bf16(hi[h], af[kk][0], af[kk][1], af[kk][2], af[kk][3], qh[(kk * 4 + 0) * 32], qh[(kk * 4 + 2) * 32]);
            mma_bf16(lo[h], af[kk][0], af[kk][1], af[kk][2], af[kk][3], qh[(kk * 4 + 1) * 32], qh[(kk * 4 + 3) * 32]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kTmMaxHeads; ++h) {
        if (h >= a.hkv) break;
        // tokens g and g + 8 of this warp's 16, tiles 2c and 2c + 1
        float m0 = fmaxf(hi[h][0] + lo[h][0], hi[h][2] + lo[h][2]);
        float m1 = fmaxf(hi[h][1] + lo[h][1], hi[h][3] + lo[h][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
        }
        if (lane < 4) {
          uint32_t* pj = part + (j * kTmMaxHeads + h) * kTpTiles;
          atomicMax(pj + 2 * c, float_to_key(m0));
          atomicMax(pj + 2 * c + 1, float_to_key(m1));
        }
      }
    }
  }
  pdl_trigger();
  __syncthreads();
  for (int i = tid; i < nblk * a.hkv * kTpTiles; i += blockDim.x) {
    const int g = i % kTpTiles, h = (i / kTpTiles) % a.hkv, j = i / (kTpTiles * a.hkv);
    const int64_t b = b0 + j;
    if (t0 + g >= t_end || b >= diag0 + g) continue;  // not a candidate of that tile
    const uint32_t u = part[(j * kTmMaxHeads + h) * kTpTiles + g];
    float m = __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
    if (rowid[j] < 0) m = -INFINITY;  // bad page: never selected
    a.scores[(static_cast<int64_t>(t0 + g) * a.hkv + h) * a.max_blocks + b] = m;
  }
}

size_t token_max_prefill_smem_bytes() {
  return 1024 + static_cast<size_t>(kTmStages) * kTmStage + kTmMaxHeads * 8 * 2 * 2 * 32 * sizeof(uint32_t) +
         static_cast<size_t>(kTpChunk) * kTmMaxHeads * kTpTiles * sizeof(uint32_t);
}

cudaError_t launch_token_max_prefill_scores(const CUtensorMap& tmi, const KvView& kv, const PrefillBatch& pb,
                                            const float* qidx, float* scores, int32_t* status, cudaStream_t stream) {
  TokenMaxPrefillArgs a;
  a.qidx = qidx;
  a.hkv = kv.hkv;
  a.max_blocks = kv.max_blocks();
  a.scores = scores;
  a.status = status;
  int64_t last = 0;  // the most candidates of any tile
  for (int s = 0; s < pb.n_seqs; ++s)
    if (pb.tile_off[s + 1] > pb.tile_off[s])
      last = max(last, pb.q_start[s] / kBlock + (pb.tile_off[s + 1] - pb.tile_off[s]) - 1);
  const int groups = pb.grp_off[pb.n_seqs];
  if (last <= 0 || groups == 0) return cudaSuccess;  // no candidates anywhere
  const unsigned chunks = static_cast<unsigned>((last + kTpChunk - 1) / kTpChunk);
  token_max_prefill_kernel<<<dim3(chunks, groups), kTmThreads, token_max_prefill_smem_bytes(), stream>>>(tmi, kv, a,
                                                                                                          pb);
  return cudaGetLastError();
}

size_t token_max_smem_bytes() { return 1024 + static_cast<size_t>(kTmStages) * kTmStage; }

cudaError_t set_token_max_smem() {
  cudaError_t e = cudaFuncSetAttribute(token_max_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(token_max_smem_bytes()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(token_max_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(token_max_prefill_smem_bytes()));
}

cudaError_t launch_token_max_scores(const CUtensorMap& tmi, const KvView& kv, int batch, const __nv_bfloat16* q,
                                    int hq, int force_local, float* scores, int32_t* status, cudaStream_t stream) {
  TokenMaxArgs a;
  a.q = q;
  a.hq = hq;
  a.hkv = kv.hkv;
  a.grp = hq / kv.hkv;
  a.force_local = force_local;
  a.max_blocks = kv.max_blocks();
  a.scores = scores;
  a.status = status;
  // one wave: the batch's blocks spread evenly over the resident CTAs
  int num_sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * kTmCtasPerSm;
  int64_t chunk = (static_cast<int64_t>(batch) * a.max_blocks + slots - 1) / slots;
  chunk = chunk < 8 ? 8 : chunk > kTmMaxChunk ? kTmMaxChunk : chunk;
  a.chunk = static_cast<int>(chunk);
  const unsigned chunks = static_cast<unsigned>((a.max_blocks + chunk - 1) / chunk);
  token_max_score_kernel<<<dim3(chunks, batch), kTmThreads, token_max_smem_bytes(), stream>>>(tmi, kv, a);
  return cudaGetLastError();
}

}  // namespace msa
