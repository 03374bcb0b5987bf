// One decode step in one kernel: Step 1 (block scores and top-k) and Step 2
// (softmax attention over the selected blocks) of the "MiniMax goes sparse"
// design (§1, Step 1 and Step 2), for a contiguous bf16 cache.
//
// A thread-block cluster of C CTAs serves one (sequence, KV head) unit; no
// CTA ever synchronises through global memory:
//   1. CTA r scores candidate blocks [r*chunk, (r+1)*chunk): a producer warp
//      streams the summary rows (bulk copies, 128 rows per 32 KB stage, a
//      3-stage ring) and eight warps dot them with the group's index query;
//      the CTA keeps its best 64 (block_select).
//   2. The leader (rank 0) gathers the C lists through distributed shared
//      memory, selects the unit's top-k, writes the index list, and leaves it
//      in its shared memory where every CTA reads its slice.
//   3. CTA r attends over its slice: the producer streams each 64x128 K and V
//      block with 2-D TMA copies (128-byte swizzle) into the 3-stage ring;
//      warps 0-3 consume every block in order (each warp 16 tokens: S = K Q^T
//      and O^T += V^T P^T on mma.sync, online softmax in fp32). Consuming in
//      order keeps each warp at most one ring cycle ahead of a slot, so a
//      parity wait can never match a stale phase.
//   4. The C partial results (m, l, O) are combined through distributed
//      shared memory: CTA r writes output pieces r, r + C, ...
#include <float.h>

#include "kernels.cuh"
#include "rows.cuh"
#include "topk64.cuh"

namespace msa {

namespace {

constexpr int kStWarps = 8;                     // compute warps
constexpr int kStThreads = 32 * (kStWarps + 1);  // + producer warp
constexpr int kStStages = 3;
constexpr int kStStage = 32768;
constexpr int kStRowsPerStage = kStStage / (kHeadDim * 2);  // 128 bf16 summary rows
constexpr int kStMaxChunk = 1024;                           // candidate rows per CTA
constexpr int kStMaxList = 64;                              // selected blocks per CTA
constexpr int kStMaxCluster = 16;
constexpr int kStG = 8;                                     // heads per group handled
constexpr int kStOS = kHeadDim + 4;                         // padded merge rows
// offsets inside the ring while it is not streaming
constexpr int kOffScratch = 0;          // SelectScratch (the selection)
constexpr int kOffFallback = 16384;     // block_topk work space (<= 16 KB)
constexpr int kOffXList = 65536;        // this CTA's best keys, read by the leader
constexpr int kOffFinal = 65536 + 512;  // the leader's final list, read by every CTA
constexpr size_t kStSmem = 1024 + kStStages * kStStage + kStMaxChunk * sizeof(uint64_t);

}  // namespace

struct StepArgs {
  const __nv_bfloat16* q;       // [batch, hq, 128]
  const __nv_bfloat16* pooled;  // [batch, hkv, max_blocks, 128]
  int hq, hkv, grp;
  int k_scored, k_total, force_local;
  int chunk;  // candidate rows per CTA, a multiple of 128, <= kStMaxChunk
  int bps;    // index-list entries attended per CTA, <= kStMaxList
  float scale_log2;
  int32_t* idx_out;  // [batch, hkv, k_total]
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
};

// grid (C, Hkv, batch), cluster (C, 1, 1).
__global__ void __launch_bounds__(kStThreads, 2) decode_step_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv, KvView kv,
                                                                   StepArgs a) {
  extern __shared__ __align__(1024) uint8_t st_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(st_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* keys = reinterpret_cast<uint64_t*>(ring + kStStages * kStStage);  // [kStMaxChunk]
  __shared__ uint64_t full[kStStages], empty[kStStages];
  __shared__ uint64_t top[64];
  __shared__ int32_t blocks[kStMaxList];
  __shared__ int sorted_blocks[64];
  __shared__ int n_blocks, count;
  __shared__ float wm[kStWarps][kStG], wl[kStWarps][kStG];

  const int rank = blockIdx.x, C = gridDim.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = static_cast<int64_t>(s) * a.hkv + h;
  const int64_t max_blocks = kv.max_tokens / kBlock;

  if (tid == 0) {
    for (int i = 0; i < kStStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kStWarps);
    }
    fence_mbar_init();
  }
  if (warp == kStWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  pdl_wait();
  const int64_t len = kv.seq_len(s, a.status, kIdDecode);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  const int64_t nbf = len / kBlock;
  int64_t n_cand = a.force_local ? min(nbf, nb - 1) : nbf;
  if (n_cand < 0) n_cand = 0;
  const int64_t forced = (a.force_local && nb > 0) ? nb - 1 : -1;
  const int64_t r0 = static_cast<int64_t>(rank) * a.chunk;
  const int rows = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.chunk), n_cand - r0)));
  const int n_st = (rows + kStRowsPerStage - 1) / kStRowsPerStage;
  __syncthreads();

  // ---------------------------------------------------------------- 1. scores
  if (warp == kStWarps) {
    if (lane == 0) {
      const __nv_bfloat16* base = a.pooled + (unit * max_blocks + r0) * kHeadDim;
      for (int st = 0; st < n_st; ++st) {
        const int slot = st % kStStages;
        if (st >= kStStages && !mbar_wait(&empty[slot], ((st / kStStages) - 1) & 1, a.status, kIdDecode)) break;
        const int n = min(kStRowsPerStage, rows - st * kStRowsPerStage);
        mbar_arrive_expect_tx(&full[slot], n * kHeadDim * 2);
        bulk_load(ring + slot * kStStage, base + static_cast<int64_t>(st) * kStRowsPerStage * kHeadDim,
                  n * kHeadDim * 2, &full[slot]);
      }
    }
  } else {
    const int e = tid & 15, hw = tid >> 4;  // 16 half-warps; lane e owns dims [8e, 8e+8)
    float qi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qi[i] = 0.f;
    for (int g = 0; g < a.grp; ++g) {
      float x[8];
      load8<__nv_bfloat16>(a.q + (static_cast<int64_t>(s) * a.hq + h * a.grp + g) * kHeadDim + 8 * e, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) qi[i] += x[i];
    }
    for (int st = 0; st < n_st; ++st) {
      const int slot = st % kStStages;
      if (!mbar_wait(&full[slot], (st / kStStages) & 1, a.status, kIdDecode)) break;
      const uint8_t* stage = ring + slot * kStStage;
      const int n = min(kStRowsPerStage, rows - st * kStRowsPerStage);
#pragma unroll
      for (int rr = 0; rr < kStRowsPerStage / 16; ++rr) {
        const int i = rr * 16 + hw;
        float part = i < n ? SelRow<__nv_bfloat16>::dot(stage + i * kHeadDim * 2, e, qi) : 0.f;
        part += __shfl_xor_sync(0xffffffffu, part, 8);
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        if (e == 0 && i < n) keys[st * kStRowsPerStage + i] = sel_key(part, static_cast<int>(r0 + st * kStRowsPerStage + i));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
  }
  __syncthreads();  // every stage consumed: the ring is free until the attention phase

  // ---------------------------------------------------------------- 2. selection
  SelectScratch& scr = *reinterpret_cast<SelectScratch*>(ring + kOffScratch);
  uint8_t* fallback = ring + kOffFallback;
  uint64_t* xlist = reinterpret_cast<uint64_t*>(ring + kOffXList);
  int32_t* final_list = reinterpret_cast<int32_t*>(ring + kOffFinal);
  const int kk = static_cast<int>(n_cand < a.k_scored ? n_cand : static_cast<int64_t>(a.k_scored));
  const int kk_local = min(kk, rows);
  if (kk_local > 0) {
    if (!block_select(keys, rows, kk_local, top, scr))
      block_topk(keys, rows, kk_local, reinterpret_cast<uint64_t*>(fallback), top, &count);
  }
  if (tid < 64) xlist[tid] = tid < kk_local ? top[tid] : 0ull;
  cluster_sync();
  if (rank == 0) {
    const int n_all = C * 64;
    for (int i = tid; i < n_all; i += blockDim.x)
      keys[i] = ld_dsmem_u64(dsmem_addr(smem_u32(xlist + (i & 63)), static_cast<uint32_t>(i >> 6)));
    __syncthreads();
    if (kk > 0) {
      if (!block_select(keys, n_all, kk, top, scr))
        block_topk(keys, n_all, kk, reinterpret_cast<uint64_t*>(fallback), top, &count);
    }
    if (tid < 32) warp_sort64_blocks_asc(top, kk, sorted_blocks);
    __syncthreads();
    int32_t* out = a.idx_out + unit * a.k_total;
    for (int i = tid; i < a.k_total; i += blockDim.x) {
      int v;
      if (i < kk) v = sorted_blocks[i];
      else if (i == kk && forced >= 0) v = static_cast<int>(forced);
      else v = -1;
      out[i] = v;
      final_list[i] = v;
    }
  }
  cluster_sync();
  if (warp == 0) {
    // this CTA's slice of the leader's list
    const uint32_t fl = dsmem_addr(smem_u32(final_list), 0u);
    const int lo = rank * a.bps, hi = min(a.k_total, lo + a.bps);
    int n = 0;
    for (int b0 = lo; b0 < hi; b0 += 32) {
      const int i = b0 + lane;
      const int32_t b = i < hi ? ld_dsmem_i32(fl + 4u * i) : -1;
      if (b >= nb) set_status(a.status, MSA_ERR_DEVICE_BOUNDS, kIdDecode);
      const bool ok = b >= 0 && b < nb;
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) blocks[n + __popc(m & ((1u << lane) - 1u))] = b;
      n += __popc(m);
    }
    if (lane == 0) n_blocks = n;
  }
  cluster_sync();  // the leader's list has been read: its ring may be reused
  if (tid == 0) {
    for (int i = 0; i < kStStages; ++i) {
      mbar_inval(&full[i]);
      mbar_inval(&empty[i]);
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);  // one warp quartet consumes each block
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int nblk = n_blocks;

  // ---------------------------------------------------------------- 3. attention
  const int g = lane >> 2, c = lane & 3;
  const int wq = warp & 3;  // token quarter of each block
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  if (warp == kStWarps) {
    if (lane == 0) {
      for (int i = 0; i < nblk; ++i) {
        const int slot = i % kStStages;
        if (i >= kStStages && !mbar_wait(&empty[slot], ((i / kStStages) - 1) & 1, a.status, kIdDecode)) break;
        const int64_t row = kv.block_row(s, h, blocks[i], a.status, kIdDecode);
        const int32_t y = static_cast<int32_t>(row < 0 ? 0 : row);
        uint8_t* dst = ring + slot * kStStage;
        mbar_arrive_expect_tx(&full[slot], kStStage);
        tma_load_2d(dst, &tmk, 0, y, &full[slot]);
        tma_load_2d(dst + 8192, &tmk, 64, y, &full[slot]);
        tma_load_2d(dst + 16384, &tmv, 0, y, &full[slot]);
        tma_load_2d(dst + 24576, &tmv, 64, y, &full[slot]);
      }
    }
  } else if (warp < 4) {
    uint32_t qb[8][2];
    {
      const bool live = g < a.grp;
      const __nv_bfloat16* qrow = a.q + (static_cast<int64_t>(s) * a.hq + h * a.grp + (live ? g : 0)) * kHeadDim;
#pragma unroll
      for (int kk2 = 0; kk2 < 8; ++kk2) {
        qb[kk2][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk2 + 2 * c) : 0u;
        qb[kk2][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk2 + 2 * c + 8) : 0u;
      }
    }
    const int krow = 16 * wq + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kchunk = lane >> 4;
    const int vrow = 16 * wq + (lane & 7) + ((lane >> 4) & 1) * 8;
    const int vchunk = (lane >> 3) & 1;
    for (int i = 0; i < nblk; ++i) {
      const int slot = i % kStStages;
      if (!mbar_wait(&full[slot], (i / kStStages) & 1, a.status, kIdDecode)) break;
      const uint32_t kbase = smem_u32(ring + slot * kStStage);
      const uint32_t vbase = kbase + 16384;
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk2 = 0; kk2 < 8; ++kk2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + (kk2 >> 2) * 8192 + swz128(krow, (kk2 & 3) * 2 + kchunk), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qb[kk2][0], qb[kk2][1]);
      }
      const int64_t tok = static_cast<int64_t>(blocks[i]) * kBlock + 16 * wq + g;
      const bool v0 = tok < len, v1 = tok + 8 < len;
      const float s0 = v0 ? sacc[0] * a.scale_log2 : -INFINITY;
      const float s1 = v0 ? sacc[1] * a.scale_log2 : -INFINITY;
      const float s2 = v1 ? sacc[2] * a.scale_log2 : -INFINITY;
      const float s3 = v1 ? sacc[3] * a.scale_log2 : -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float rf0 = mn0 == -INFINITY ? 0.f : mn0;
      const float rf1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - rf0), al1 = exp2f(m1 - rf1);
      const float p0 = exp2f(s0 - rf0), p2 = exp2f(s2 - rf0);
      const float p1 = exp2f(s1 - rf1), p3 = exp2f(s3 - rf1);
      l0 = l0 * al0 + p0 + p2;
      l1 = l1 * al1 + p1 + p3;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o[j][0] *= al0; o[j][1] *= al1; o[j][2] *= al0; o[j][3] *= al1;
      }
      const uint32_t pb0 = movm_t(pack_bf16(p0, p1));
      const uint32_t pb1 = movm_t(pack_bf16(p2, p3));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + (j >> 2) * 8192 + swz128(vrow, (j & 3) * 2 + vchunk), a0, a1, a2, a3);
        mma_bf16(o[j], a0, a1, a2, a3, pb0, pb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
  pdl_trigger();
  __syncthreads();  // the ring is free again: warp states go there
  float* obuf = reinterpret_cast<float*>(ring);                        // [8 warps][8 heads][132]
  float* xch = obuf + kStWarps * kStG * kStOS;                         // M[8], L[8], O[8][128]
  if (warp < kStWarps) {
    float* ob = obuf + warp * kStG * kStOS;
    if (g == 0) {
      wm[warp][2 * c] = m0;
      wm[warp][2 * c + 1] = m1;
      wl[warp][2 * c] = l0;
      wl[warp][2 * c + 1] = l1;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ob[(2 * c) * kStOS + 16 * j + g] = o[j][0];
      ob[(2 * c + 1) * kStOS + 16 * j + g] = o[j][1];
      ob[(2 * c) * kStOS + 16 * j + g + 8] = o[j][2];
      ob[(2 * c + 1) * kStOS + 16 * j + g + 8] = o[j][3];
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- 4. combine
  {
    const int head = tid >> 4, d0 = (tid & 15) * 8;
    if (tid < 128 && head < a.grp) {
      float M = -INFINITY;
      for (int w = 0; w < kStWarps; ++w) M = fmaxf(M, wm[w][head]);
      float L = 0.f, acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < kStWarps; ++w) {
          const float f = exp2f(wm[w][head] - M);
          L += f * wl[w][head];
          const float* src = obuf + (w * kStG + head) * kStOS + d0;
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(f, src[i], acc[i]);
        }
      }
      if (C == 1) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
        uint4 v;
        v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        v.z = pack_bf16(acc[4] * inv, acc[5] * inv);
        v.w = pack_bf16(acc[6] * inv, acc[7] * inv);
        const int64_t qrow = static_cast<int64_t>(s) * a.hq + h * a.grp + head;
        *reinterpret_cast<uint4*>(a.out + qrow * kHeadDim + d0) = v;
        if (a.lse != nullptr && d0 == 0) a.lse[qrow] = L > 0.f ? M * kLn2 + logf(L) : -INFINITY;
      } else {
        if (d0 == 0) {
          xch[head] = M;
          xch[kStG + head] = L;
        }
        float* dst = xch + 2 * kStG + head * kHeadDim + d0;
        reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
  }
  if (C == 1) return;
  cluster_sync();
  if (tid < 128) {
    const int n = C;
    const int pieces = a.grp * 16;
    const int j = tid / n, i = tid % n;
    const int piece = j * n + rank;
    const bool live = piece < pieces;
    const int head = live ? piece >> 4 : 0;
    const int d0 = live ? (piece & 15) * 8 : 0;
    float Mi = -INFINITY, Li = 0.f;
    float4 oa = make_float4(0.f, 0.f, 0.f, 0.f), ob = oa;
    if (live) {
      const uint32_t base = dsmem_addr(smem_u32(xch), static_cast<uint32_t>(i));
      Mi = ld_dsmem(base + 4u * head);
      Li = ld_dsmem(base + 4u * (kStG + head));
      oa = ld_dsmem4(base + 4u * (2 * kStG + head * kHeadDim + d0));
      ob = ld_dsmem4(base + 4u * (2 * kStG + head * kHeadDim + d0 + 4));
    }
    float Mx = Mi;
    for (int off = n >> 1; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
    const float f = (Mx == -INFINITY) ? 0.f : exp2f(Mi - Mx);
    float v[9] = {f * Li, f * oa.x, f * oa.y, f * oa.z, f * oa.w, f * ob.x, f * ob.y, f * ob.z, f * ob.w};
    for (int off = n >> 1; off > 0; off >>= 1) {
#pragma unroll
      for (int q = 0; q < 9; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], off);
    }
    if (live && i == 0) {
      const float inv = v[0] > 0.f ? 1.f / v[0] : 0.f;
      uint4 w;
      w.x = pack_bf16(v[1] * inv, v[2] * inv);
      w.y = pack_bf16(v[3] * inv, v[4] * inv);
      w.z = pack_bf16(v[5] * inv, v[6] * inv);
      w.w = pack_bf16(v[7] * inv, v[8] * inv);
      const int64_t qrow = static_cast<int64_t>(s) * a.hq + h * a.grp + head;
      *reinterpret_cast<uint4*>(a.out + qrow * kHeadDim + d0) = w;
      if (a.lse != nullptr && d0 == 0) a.lse[qrow] = v[0] > 0.f ? Mx * kLn2 + logf(v[0]) : -INFINITY;
    }
  }
  cluster_sync();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Cluster shape of the fused step, or false when it does not apply (then the
// step runs as the two separate kernels). C is a power of two <= 16 with
// units x C within two resident CTAs per SM, chunk = ceil(max_blocks / C)
// rounded up to 128 rows (<= 1024), and ceil(k_total / C) <= 64 list entries.
bool step_shape(int64_t units, int64_t max_blocks, int k_scored, int k_total, int num_sms, int* C, int* chunk,
                int* bps) {
  if (k_scored > 64) return false;
  const int64_t slots = 2LL * num_sms;
  int c = 1;
  while (c < kStMaxCluster && units * c * 2 <= slots) c *= 2;
  while (c < kStMaxCluster && ((max_blocks + c - 1) / c > kStMaxChunk || (k_total + c - 1) / c > kStMaxList)) c *= 2;
  int64_t ch = (max_blocks + c - 1) / c;
  ch = (ch + kStRowsPerStage - 1) / kStRowsPerStage * kStRowsPerStage;
  if (ch > kStMaxChunk || (k_total + c - 1) / c > kStMaxList) return false;
  *C = c;
  *chunk = static_cast<int>(ch);
  *bps = (k_total + c - 1) / c;
  return true;
}

cudaError_t set_step_smem() {
  cudaError_t e = cudaFuncSetAttribute(decode_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kStSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_step_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_step_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

cudaError_t launch_decode_step(const CUtensorMap& tmk, const CUtensorMap& tmv, const KvView& kv, int batch,
                               const __nv_bfloat16* q, int hq, const __nv_bfloat16* pooled,
                               const msa_select_cfg& cfg, int k_total, int C, int chunk, int bps, float scale_log2,
                               int32_t* idx_out, __nv_bfloat16* out, float* lse, int32_t* status,
                               cudaStream_t stream) {
  StepArgs a;
  a.q = q;
  a.pooled = pooled;
  a.hq = hq;
  a.hkv = kv.hkv;
  a.grp = hq / kv.hkv;
  a.k_scored = cfg.k_scored;
  a.k_total = k_total;
  a.force_local = cfg.force_local;
  a.chunk = chunk;
  a.bps = bps;
  a.scale_log2 = scale_log2;
  a.idx_out = idx_out;
  a.out = out;
  a.lse = lse;
  a.status = status;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(C, kv.hkv, batch);
  lc.blockDim = dim3(kStThreads, 1, 1);
  lc.dynamicSmemBytes = kStSmem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, decode_step_kernel, tmk, tmv, kv, a);
}

}  // namespace msa
