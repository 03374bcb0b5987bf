// One decode step in one kernel: Step 1 (block scores and top-k) and Step 2
// (softmax attention over the selected blocks) of the "MiniMax goes sparse"
// design (§1, Step 1 and Step 2), for a contiguous bf16 cache.
//
// A thread-block cluster of C CTAs serves one (sequence, KV head) unit; no
// CTA ever synchronises through global memory:
//   1. CTA r scores candidate blocks [r*chunk, (r+1)*chunk): a producer warp
//      streams the summary rows (2-D TMA, 128 rows per 32 KB stage, a 3-stage
//      ring) and eight warps dot them with the group's index query on the
//      tensor cores (mma.sync, the query split into two bf16 parts).
//   2. Selection in two cluster exchanges, exact by construction: each warp
//      offers the running maxima of its keys as samples; the k-th largest
//      sample score L bounds the unit's k-th score from below, so each CTA
//      keeps only its keys scoring >= L; every CTA then gathers that small
//      union through distributed shared memory and ranks it, so each holds
//      the unit's top-k and takes its slice of the list (the leader writes
//      the list out, sorted, while the attention runs). A union too large
//      for this (e.g. every score equal) takes an exact radix-select path.
//   3. CTA r attends over its slice: the producer streams each 64x128 K and V
//      block with 2-D TMA copies (128-byte swizzle) into the 3-stage ring;
//      warps 0-3 consume every block in order (each warp 16 tokens: S = K Q^T
//      and O^T += V^T P^T on mma.sync, online softmax in fp32). Consuming in
//      order keeps each warp at most one ring cycle ahead of a slot, so a
//      parity wait can never match a stale phase.
//   4. The C partial results (m, l, O) are combined through distributed
//      shared memory: every CTA pushes piece p (one head, 8 dims) of its
//      partial into the shared memory of CTA p % C, and after one cluster
//      barrier CTA r merges and writes output pieces r, r + C, ...
// With scores computed apart (the token-max scores of the guide's Step 1 as
// drawn, by the kernel before this one), phase 1 reads each CTA's chunk of
// block scores instead of streaming and scoring summary rows; phases 2-4 are
// the same.
#include <float.h>

#include <algorithm>

#include "kernels.cuh"
#include "rows.cuh"
#include "topk64.cuh"

namespace msa {

namespace {

constexpr int kStWarps = 8;                     // compute warps
constexpr int kStAttnWarps = 4;                 // warps that consume attention blocks
constexpr int kStThreads = 32 * (kStWarps + 1);  // + producer warp
constexpr int kStStages = 3;                    // ring depth (two CTAs per SM)
constexpr int kStStage = 32768;
constexpr int kStRowsPerStage = kStStage / (kHeadDim * 2);  // 128 bf16 summary rows
constexpr int kStMaxChunk = 1024;                           // candidate rows per CTA
constexpr int kStMaxList = 64;                              // selected blocks per CTA
constexpr int kStMaxCluster = 16;
constexpr int kStG = 8;                                     // heads per group handled
constexpr int kStOS = kHeadDim + 4;                         // padded merge rows
constexpr int kStRecv = 12;                                 // floats per pushed piece: O[8], M, L, pad
constexpr size_t step_smem(int stages) { return 1024 + stages * kStStage + kStMaxChunk * sizeof(uint64_t); }

}  // namespace

struct StepArgs {
  const __nv_bfloat16* q;       // [batch, hq, 128]
  int hq, hkv, grp;
  int k_scored, k_total, force_local;
  int chunk;  // candidate rows per CTA, a multiple of 128, <= kStMaxChunk
  int bps;    // index-list entries attended per CTA, <= kStMaxList
  int samples_per_warp;  // 1, 2, 4 or 8 sample keys per compute warp for the selection bound
  float scale_log2;
  int32_t* idx_out;  // [batch, hkv, k_total]
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  const __nv_bfloat16* k;        // keys (for pooling the newest block)
  __nv_bfloat16* pooled_out;     // nullable: summary of the newest block when it has just filled
  const float* pre_scores;       // scores computed apart: [batch, hkv, max_blocks] (kPre kernels only)
};

// grid (C, Hkv, batch), cluster (C, 1, 1). kStages: depth of the shared-memory
// ring; kPre: the block scores come from a.pre_scores.
template <int kStages, bool kPre>
__global__ void __launch_bounds__(kStThreads, 2) decode_step_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv,
                                                                   const __grid_constant__ CUtensorMap tmpool, KvView kv,
                                                                   StepArgs a) {
  extern __shared__ __align__(1024) uint8_t st_raw[];
  uint8_t* ring = smem_align1024(st_raw);  // keys and the selection buffers follow in shared memory
  uint64_t* keys = reinterpret_cast<uint64_t*>(ring + kStages * kStStage);  // [kStMaxChunk]
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ uint64_t xlist2[64];    // exact path: this CTA's best kk keys
  __shared__ uint32_t xsamp[64];     // this CTA's sample scores (read by the cluster)
  __shared__ uint64_t xsurv[64];     // this CTA's keys scoring >= L (read by the cluster)
  __shared__ uint32_t lbound;
  __shared__ int ccount[kStMaxCluster];
  __shared__ uint64_t sel_keys[64];  // the unit's selected keys
  __shared__ RadixScratch radix;
  __shared__ int n_sel;   // this CTA's survivor count (may exceed 64: then only 64 are stored)
  __shared__ int n_sel2;  // counter of the exact path
  __shared__ float qsum[kHeadDim];  // the group's index query (sum of its query heads), fp32
  __shared__ float wm[kStAttnWarps][kStG], wl[kStAttnWarps][kStG];

  const int rank = blockIdx.x, C = gridDim.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = static_cast<int64_t>(s) * a.hkv + h;
  const int64_t max_blocks = kv.max_blocks();  // summary rows per unit

  // The producer sets up the ring and, as soon as the inputs are ready, starts
  // streaming the first stages of its chunk: their rows do not depend on the
  // sequence length, which is read meanwhile (stages past the candidates are
  // drained unread).
  const int n_pre = kPre ? 0 : min(kStages, (a.chunk + kStRowsPerStage - 1) / kStRowsPerStage);
  const int32_t y0 = static_cast<int32_t>(unit * max_blocks + static_cast<int64_t>(rank) * a.chunk);
  if (warp == kStWarps && lane == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kStWarps);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmpool);
    // While the kernel before this one finishes, its first stages' rows are
    // pulled into L2 (a prefetch has no result: if that kernel writes any of
    // them, the loads below, issued after it has completed, read its values).
    for (int st = 0; st < n_pre; ++st) {
      tma_prefetch_2d(&tmpool, 0, y0 + st * kStRowsPerStage);
      tma_prefetch_2d(&tmpool, 64, y0 + st * kStRowsPerStage);
    }
    pdl_wait();
    for (int st = 0; st < n_pre; ++st) {
      uint8_t* dst = ring + st * kStStage;
      mbar_arrive_expect_tx(&full[st], kStStage);
      tma_load_2d(dst, &tmpool, 0, y0 + st * kStRowsPerStage, &full[st]);
      tma_load_2d(dst + kStStage / 2, &tmpool, 64, y0 + st * kStRowsPerStage, &full[st]);
    }
  }
  pdl_wait();
  if (!kPre && tid < kHeadDim) {
    // all G loads in flight at once, then summed in head order
    const __nv_bfloat16* qg = a.q + (static_cast<int64_t>(s) * a.hq + h * a.grp) * kHeadDim + tid;
    float x[kStG];
#pragma unroll
    for (int g = 0; g < kStG; ++g) x[g] = g < a.grp ? __bfloat162float(qg[g * kHeadDim]) : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int g = 0; g < kStG; ++g) acc += x[g];
    qsum[tid] = acc;
  }
  const int64_t len = kv.seq_len(s, a.status, kIdDecode);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  const int64_t nbf = len / kBlock;
  const bool local = (a.force_local & kForceLocal) != 0, sink = (a.force_local & kForceSink) != 0;
  int64_t n_cand = local ? min(nbf, nb - 1) : nbf;
  if (n_cand < 0) n_cand = 0;
  const int64_t forced = (local && nb > 0) ? nb - 1 : -1;
  const int skip = (sink && n_cand > 0) ? 1 : 0;  // attention sink: block 0 kept, not scored
  const int keep0 = (sink && nb > 0 && forced != 0) ? 1 : 0;
  const int64_t r0 = static_cast<int64_t>(rank) * a.chunk;
  const int rows = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.chunk), n_cand - r0)));
  const int n_st = kPre ? 0 : (rows + kStRowsPerStage - 1) / kStRowsPerStage;
  if (rank == 0 && warp == kStWarps && lane >= 28 && forced >= 0) {
    // the newest block is always attended: pull it into L2 during scoring
    const int64_t row = kv.block_row(s, h, forced, a.status, kIdDecode);
    if (row >= 0) tma_prefetch_2d((lane & 2) ? &tmv : &tmk, (lane & 1) * 64, static_cast<int32_t>(row));
  }
  __syncthreads();

  // ---------------------------------------------------------------- 1. scores
  uint64_t lmax = 0ull;  // compute warps: the largest key this lane produced
  if constexpr (kPre) {
    if (warp < kStWarps) {
      // this CTA's chunk of the unit's scores, every load in flight at once;
      // lanes 4j fold in the keys of lanes 4j + 1 .. 4j + 3, as the samples
      // are taken from lanes 4j
      constexpr int kPer = kStMaxChunk / (32 * kStWarps);
      const float* sc = a.pre_scores + unit * max_blocks + r0;
      float v[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = tid + 32 * kStWarps * u;
        v[u] = i < rows ? sc[i] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = tid + 32 * kStWarps * u;
        if (i < rows) {
          const uint64_t key = (skip && r0 + i == 0) ? 0ull : sel_key(v[u], static_cast<int>(r0 + i));
          keys[i] = key;
          lmax = key > lmax ? key : lmax;
        }
      }
      uint64_t o = shfl_xor_u64(lmax, 1);
      lmax = o > lmax ? o : lmax;
      o = shfl_xor_u64(lmax, 2);
      lmax = o > lmax ? o : lmax;
    }
  } else if (warp == kStWarps) {
    if (lane == 0) {
      // 128 summary rows per stage as two 64-column boxes (128-byte swizzle);
      // rows past the CTA's chunk are loaded but never scored
      int issued = n_pre;
      for (int st = n_pre; st < n_st; ++st) {
        const int slot = st % kStages;
        if (st >= kStages && !mbar_wait(&empty[slot], ((st / kStages) - 1) & 1, a.status, kIdDecode)) break;
        uint8_t* dst = ring + slot * kStStage;
        mbar_arrive_expect_tx(&full[slot], kStStage);
        tma_load_2d(dst, &tmpool, 0, y0 + st * kStRowsPerStage, &full[slot]);
        tma_load_2d(dst + kStStage / 2, &tmpool, 64, y0 + st * kStRowsPerStage, &full[slot]);
        issued = st + 1;
      }
      // every stage issued has landed, the early ones beyond this chunk's
      // candidates (never read) included, before the ring is reused
      mbar_drain(full, kStages, issued, a.status, kIdDecode);
    }
  } else {
    // S = K_pool q_idx on the tensor cores, warp w taking rows 16w..16w+15 of
    // each stage. The B operand holds the fp32 index query split into a bf16
    // head (column 0) and the bf16 of the remainder (column 1), so the two
    // accumulator columns add up to the fp32 dot product to ~2^-16 relative.
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
    const int krow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kchunk = lane >> 4;
    for (int st = 0; st < n_st; ++st) {
      const int slot = st % kStages;
      if (!mbar_wait_warp(&full[slot], (st / kStages) & 1, a.status, kIdDecode)) break;
      const uint32_t sbase = smem_u32(ring + slot * kStStage);
      const int n = min(kStRowsPerStage, rows - st * kStRowsPerStage);
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk2 = 0; kk2 < 8; ++kk2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sbase + (kk2 >> 2) * (kStStage / 2) + swz128(krow, (kk2 & 3) * 2 + kchunk), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qb[kk2][0], qb[kk2][1]);
      }
      uint64_t ka = 0ull, kb = 0ull;
      if (c == 0) {
        const int i0 = 16 * warp + g, i1 = i0 + 8;
        const int base = st * kStRowsPerStage;
        if (i0 < n) {
          ka = (skip && r0 + base + i0 == 0) ? 0ull : sel_key(sacc[0] + sacc[1], static_cast<int>(r0 + base + i0));
          keys[base + i0] = ka;
        }
        if (i1 < n) {
          kb = sel_key(sacc[2] + sacc[3], static_cast<int>(r0 + base + i1));
          keys[base + i1] = kb;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      lmax = ka > lmax ? ka : lmax;
      lmax = kb > lmax ? kb : lmax;
    }
  }
  __syncthreads();  // every stage consumed: the ring is free until the attention phase

  // ---------------------------------------------------------------- 2. selection
  // Fast path, exact by construction:
  // (a) Samples: every compute warp offers the largest key of each of its p
  //     lane groups (p per warp, chosen so the cluster holds >= 2 kk samples).
  //     The samples are real keys, so their kk-th largest score L is at most
  //     the score of the unit's kk-th key: every key of the selection scores
  //     >= L.
  // (b) After a cluster barrier every CTA gathers all samples through
  //     distributed shared memory and finds L by rank counting; it keeps its
  //     own keys scoring >= L (survivors, normally a few more than kk / C).
  // (c) After a second cluster barrier every CTA gathers all survivors and
  //     ranks them: the best kk, in rank order, are the unit's selection.
  // If a CTA has more than 64 survivors or the union more than 256 (e.g.
  // every score equal), every CTA takes the exact path instead: a radix
  // select of its own kk best keys, an exchange, and a radix select over
  // their union. The decision is the same in every CTA of the cluster.
  uint64_t* lists = reinterpret_cast<uint64_t*>(ring);  // [C][64]: gathered keys
  uint32_t* samp_all = reinterpret_cast<uint32_t*>(ring + 16384);  // [C * 8 * p] gathered sample scores
  const int kk = static_cast<int>(n_cand - skip < a.k_scored ? n_cand - skip : static_cast<int64_t>(a.k_scored));
  const int p = a.samples_per_warp;  // 1, 2, 4 or 8
  const int n_samp = kStWarps * p;
  if (warp < kStWarps) {
    // group max over the key-holding lanes (lane = 4 j, j = 0..7) of each group of 8 / p
    uint64_t v = lmax;
    for (int o = 1; o < 8 / p; o <<= 1) {
      const uint64_t w2 = shfl_xor_u64(v, 4 * o);
      v = w2 > v ? w2 : v;
    }
    const int j = lane >> 2;
    if ((lane & 3) == 0 && (j % (8 / p)) == 0) xsamp[warp * p + j / (8 / p)] = static_cast<uint32_t>(v >> 32);
  }
  __syncthreads();
  if (C > 1) cluster_arrive();
  if (warp == kStWarps && lane == 0) {
    // the ring's barriers restart for the attention phase (one warp quartet
    // consumes each block); nothing waits on them until then, and the
    // producer does this while the cluster catches up
    for (int i = 0; i < kStages; ++i) {
      mbar_inval(&full[i]);
      mbar_inval(&empty[i]);
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kStAttnWarps);
    }
    fence_mbar_init();
  }
  __syncwarp();
  if (C > 1) cluster_wait();
  for (int i = tid; i < C * n_samp; i += blockDim.x) {
    const int r = i / n_samp, j = i - r * n_samp;
    samp_all[i] = C > 1 ? static_cast<uint32_t>(ld_dsmem_i32(dsmem_addr(smem_u32(xsamp + j), static_cast<uint32_t>(r))))
                        : xsamp[j];
  }
  if (tid == 0) {
    lbound = 0u;
    n_sel = 0;
  }
  __syncthreads();
  {
    // L = the kk-th largest sample score: the value with fewer than kk samples
    // above it and at least kk at or above it (equal values write the same L).
    // q adjacent threads count for each sample and add their counts.
    const int ns = C * n_samp;  // <= 128, a multiple of 8
    const int q = ns <= 72 ? 4 : 2;
    const int i = tid / q, part = tid - i * q;
    const uint32_t v = i < ns ? samp_all[i] : 0u;
    int gt = 0, ge = 0;
    if (i < ns) {
      const uint4* s4 = reinterpret_cast<const uint4*>(samp_all);
#pragma unroll 4
      for (int j = part; j < ns / 4; j += q) {
        const uint4 u = s4[j];
        gt += (u.x > v) + (u.y > v) + (u.z > v) + (u.w > v);
        ge += (u.x >= v) + (u.y >= v) + (u.z >= v) + (u.w >= v);
      }
    }
    for (int o = 1; o < q; o <<= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      ge += __shfl_xor_sync(0xffffffffu, ge, o);
    }
    if (i < ns && part == 0 && gt < kk && kk <= ge) lbound = v;
  }
  __syncthreads();
  {
    const uint32_t L = lbound;
    for (int base = 0; base < rows; base += blockDim.x) {
      const int i = base + tid;
      const uint64_t key = i < rows ? keys[i] : 0ull;
      const bool hit = key != 0ull && static_cast<uint32_t>(key >> 32) >= L;
      const unsigned mk = __ballot_sync(0xffffffffu, hit);
      int slot = 0;
      if (lane == 0 && mk != 0u) slot = atomicAdd(&n_sel, __popc(mk));
      slot = __shfl_sync(0xffffffffu, slot, 0);
      const int pos = slot + __popc(mk & ((1u << lane) - 1u));
      if (hit && pos < 64) xsurv[pos] = key;
    }
  }
  // n_sel now holds this CTA's survivor count (read by the cluster; the exact
  // path counts with n_sel2, so it is never written again)
  __syncthreads();
  if (C > 1) cluster_arrive();
  if (C > 1) cluster_wait();
  if (tid < C) ccount[tid] = C > 1 ? ld_dsmem_i32(dsmem_addr(smem_u32(&n_sel), static_cast<uint32_t>(tid))) : n_sel;
  if (tid < 64) sel_keys[tid] = 0ull;
  __syncthreads();
  int n_union = 0, overflow = 0;
  for (int r = 0; r < C; ++r) {
    overflow |= ccount[r] > 64 ? 1 : 0;
    n_union += ccount[r];
  }
  const bool exact = kk == 0 || (!overflow && n_union <= 256 && n_union >= kk);
  if (exact && kk > 0) {
    for (int i = tid; i < n_union; i += blockDim.x) {
      int r = 0, off = i;
      while (off >= ccount[r]) off -= ccount[r++];
      lists[i] = C > 1 ? ld_dsmem_u64(dsmem_addr(smem_u32(xsurv + off), static_cast<uint32_t>(r))) : xsurv[off];
    }
    if (tid == 0) lists[n_union] = 0ull;
    __syncthreads();
    // rank counting, q adjacent threads per key: the best kk go to sel_keys in rank order
    const int q = n_union <= 72 ? 4 : (n_union <= 144 ? 2 : 1);
    const int i = tid / q, part = tid - i * q;
    const uint64_t x = i < n_union ? lists[i] : 0ull;
    int cnt = 0;
    if (i < n_union) {
      const ulonglong2* l2 = reinterpret_cast<const ulonglong2*>(lists);  // lists[n_union] is 0 (padding)
#pragma unroll 4
      for (int j = part; j < (n_union + 1) / 2; j += q) {
        const ulonglong2 y = l2[j];
        cnt += (y.x > x) + (y.y > x);
      }
    }
    for (int o = 1; o < q; o <<= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (i < n_union && part == 0 && cnt < kk) sel_keys[cnt] = x;
  } else if (!exact) {
    // exact path: this CTA's kk best keys by radix select, a second exchange,
    // and a radix select over their union
    if (tid < 64) xlist2[tid] = 0ull;
    const uint64_t t_local = block_kth_largest(keys, rows, kk, radix);
    block_compact_ge(keys, rows, t_local, xlist2, 64, &n_sel2);
    if (C > 1) cluster_sync();
    for (int i = tid; i < C * 64; i += blockDim.x)
      lists[i] = C > 1 ? ld_dsmem_u64(dsmem_addr(smem_u32(xlist2 + (i & 63)), static_cast<uint32_t>(i >> 6)))
                       : xlist2[i];
    __syncthreads();
    const uint64_t t_unit = block_kth_largest(lists, C * 64, kk, radix);
    uint64_t* picked = lists + 1024;  // past the C * 64 gathered keys
    block_compact_ge(lists, C * 64, t_unit, picked, 64, &n_sel2);
    // rank order (the compaction's order differs between CTAs)
    if (tid < kk) {
      const uint64_t x = picked[tid];
      int cnt = 0;
      for (int j = 0; j < kk; ++j) cnt += picked[j] > x ? 1 : 0;
      sel_keys[cnt] = x;
    }
  }
  __syncthreads();
  // (c) the unit's list. Attention slices use the rank order (the same in
  // every CTA of the cluster): block 0 first when kept as the attention sink,
  // then the kk selected blocks, then the forced newest block, then -1. The
  // leader writes the list sorted ascending to idx_out while the attention
  // runs (warps 5-7 are idle then).
  auto slice_at = [&](int i) -> int32_t {
    const int j = i - keep0;
    return j < 0 ? 0 : j < kk ? sel_block(sel_keys[j]) : (j == kk && forced >= 0 ? static_cast<int32_t>(forced) : -1);
  };
  // The list's valid entries are a prefix (block 0, the kk blocks, the newest
  // block; -1 after them), so this CTA's slice needs no compaction: every
  // thread knows its length and reads its entries straight from sel_keys.
  const int lo = rank * a.bps, hi = min(a.k_total, lo + a.bps);
  const int n_valid = keep0 + kk + (forced >= 0 ? 1 : 0);
  const int nblk = max(0, min(hi, n_valid) - lo);

  // ---------------------------------------------------------------- 3. attention
  const int g = lane >> 2, c = lane & 3;
  const int wq = warp & 3;  // token quarter of each block (attention warps 0-3)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  if (warp == kStWarps) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        const int slot = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[slot], ((i / kStages) - 1) & 1, a.status, kIdDecode)) break;
        issued = i + 1;
        const int32_t b = slice_at(lo + i);
        if (b >= nb) set_status(a.status, MSA_ERR_DEVICE_BOUNDS, kIdDecode);  // its keys are masked below
        const int64_t row = b < nb ? kv.block_row(s, h, b, a.status, kIdDecode) : -1;
        const int32_t y = static_cast<int32_t>(row < 0 ? 0 : row);
        uint8_t* dst = ring + slot * kStStage;
        mbar_arrive_expect_tx(&full[slot], kStStage);
        tma_load_2d(dst, &tmk, 0, y, &full[slot]);
        tma_load_2d(dst + 8192, &tmk, 64, y, &full[slot]);
        tma_load_2d(dst + 16384, &tmv, 0, y, &full[slot]);
        tma_load_2d(dst + 24576, &tmv, 64, y, &full[slot]);
      }
      mbar_drain(full, kStages, issued, a.status, kIdDecode);
    }
  } else if (warp < kStAttnWarps) {
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
      const int slot = i % kStages;
      if (!mbar_wait_warp(&full[slot], (i / kStages) & 1, a.status, kIdDecode)) break;
      const uint32_t kbase = smem_u32(ring + slot * kStStage);
      const uint32_t vbase = kbase + 16384;
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk2 = 0; kk2 < 8; ++kk2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + (kk2 >> 2) * 8192 + swz128(krow, (kk2 & 3) * 2 + kchunk), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qb[kk2][0], qb[kk2][1]);
      }
      const int64_t tok = static_cast<int64_t>(slice_at(lo + i)) * kBlock + 16 * wq + g;
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
  } else if (warp > kStAttnWarps && rank == 0) {
    // warps 5-7 of the leader: the unit's list, ascending (block 0 when kept as
    // the sink, the kk selected blocks by counting -- each one's position is
    // the number of selected blocks below it -- the newest block, then -1)
    const int t = tid - 32 * (kStAttnWarps + 1);
    int32_t* out = a.idx_out + unit * a.k_total;
    if (t < kk) {
      const int b = sel_block(sel_keys[t]);
      int pos = 0;
      for (int j = 0; j < kk; ++j) pos += sel_block(sel_keys[j]) < b ? 1 : 0;
      out[keep0 + pos] = b;
    }
    for (int i = t; i < a.k_total; i += 32 * (kStWarps - kStAttnWarps - 1)) {
      if (i >= keep0 && i < keep0 + kk) continue;
      out[i] = (i < keep0) ? 0 : (i == keep0 + kk && forced >= 0 ? static_cast<int32_t>(forced) : -1);
    }
  } else if (warp == kStAttnWarps && lane < 16 && rank == 0 && a.pooled_out != nullptr && forced >= 0 &&
             len % kBlock == 0) {
    // While warps 0-3 attend, the leader's first idle half-warp writes the
    // summary of the newest block, which has just filled: the next step scores
    // it. Same arithmetic as the pooling kernel (fp32 sum of the 64 rows in
    // order, one multiply by 1/64, round to nearest even); lane e owns dims
    // [8e, 8e + 8). The rows are in L2 (prefetched at the start).
    const int64_t row = kv.block_row(s, h, forced, a.status, kIdDecode);
    if (row >= 0) {
      const uint4* src = reinterpret_cast<const uint4*>(a.k + row * kHeadDim) + lane;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 1
      for (int t0 = 0; t0 < kBlock; t0 += 16) {
        uint4 v[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) v[t] = __ldg(src + (t0 + t) * (kHeadDim / 8));
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
          }
        }
      }
      uint4 o;
      o.x = pack_bf16(acc[0] * (1.0f / kBlock), acc[1] * (1.0f / kBlock));
      o.y = pack_bf16(acc[2] * (1.0f / kBlock), acc[3] * (1.0f / kBlock));
      o.z = pack_bf16(acc[4] * (1.0f / kBlock), acc[5] * (1.0f / kBlock));
      o.w = pack_bf16(acc[6] * (1.0f / kBlock), acc[7] * (1.0f / kBlock));
      *reinterpret_cast<uint4*>(a.pooled_out + (unit * max_blocks + forced) * kHeadDim + 8 * lane) = o;
    }
  }
  pdl_trigger();
  __syncthreads();  // the ring is free again: warp states go there
  float* obuf = reinterpret_cast<float*>(ring);  // [4 warps][8 heads][132]
  float* recv = reinterpret_cast<float*>(keys);  // [C][128 / C][kStRecv]: pieces pushed by the cluster
  if (warp < kStAttnWarps) {
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
      for (int w = 0; w < kStAttnWarps; ++w) M = fmaxf(M, wm[w][head]);
      float L = 0.f, acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < kStAttnWarps; ++w) {
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
        // push this CTA's part of piece `tid` (head, 8 dims) to the piece's
        // owner, rank tid % C: slot [rank][tid / C] of the owner's receive
        // area, which (like all of `keys`) is free once the owner has passed
        // the selection barrier, as every CTA pushing here has
        const uint32_t dst = dsmem_addr(smem_u32(recv + (rank * (128 / C) + tid / C) * kStRecv),
                                        static_cast<uint32_t>(tid % C));
        st_dsmem4(dst, make_float4(acc[0], acc[1], acc[2], acc[3]));
        st_dsmem4(dst + 16u, make_float4(acc[4], acc[5], acc[6], acc[7]));
        st_dsmem4(dst + 32u, make_float4(M, L, 0.f, 0.f));
      }
    }
  }
  if (C == 1) return;
  // every piece has arrived; after this no CTA touches another's shared memory
  cluster_sync();
  if (tid < 128) {
    const int n = C;
    const int pieces = a.grp * 16;
    const int j = tid / n, i = tid % n;  // owned slot j, from rank i
    const int piece = j * n + rank;
    const bool live = piece < pieces;
    const int head = live ? piece >> 4 : 0;
    const int d0 = live ? (piece & 15) * 8 : 0;
    float Mi = -INFINITY, Li = 0.f;
    float4 oa = make_float4(0.f, 0.f, 0.f, 0.f), ob = oa;
    if (live) {
      const float* src = recv + (i * (128 / n) + j) * kStRecv;
      oa = *reinterpret_cast<const float4*>(src);
      ob = *reinterpret_cast<const float4*>(src + 4);
      const float4 ml = *reinterpret_cast<const float4*>(src + 8);
      Mi = ml.x;
      Li = ml.y;
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
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Cluster shape of the fused step, or false when it does not apply (then the
// step runs as the two separate kernels). C is a power of two <= 16 with
// units x C within two resident CTAs per SM and, where max_clusters is given
// (the device's co-resident cluster count for C = 1, 2, 4, 8, 16), every
// unit's cluster resident at once; chunk = ceil(max_blocks / C) rounded up to
// 128 rows (<= 1024), and ceil(k_total / C) <= 64 list entries.
bool step_shape(int64_t units, int64_t max_blocks, int k_scored, int k_total, int num_sms, const int* max_clusters,
                int* C, int* chunk, int* bps) {
  if (k_scored > 64) return false;
  const int64_t slots = 2LL * num_sms;
  int c = 1, lg = 0;
  while (c < kStMaxCluster && units * c * 2 <= slots && (max_clusters == nullptr || units <= max_clusters[lg + 1])) {
    c *= 2;
    ++lg;
  }
  while (c < kStMaxCluster && ((max_blocks + c - 1) / c > kStMaxChunk || (k_total + c - 1) / c > kStMaxList)) {
    c *= 2;
    ++lg;
  }
  int64_t ch = (max_blocks + c - 1) / c;
  ch = (ch + kStRowsPerStage - 1) / kStRowsPerStage * kStRowsPerStage;
  if (ch > kStMaxChunk || (k_total + c - 1) / c > kStMaxList) return false;
  *C = c;
  *chunk = static_cast<int>(ch);
  *bps = (k_total + c - 1) / c;
  return true;
}

namespace {

template <int kStages>
int max_clusters_of(int C) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, 1, 1);
  cfg.blockDim = dim3(kStThreads, 1, 1);
  cfg.dynamicSmemBytes = step_smem(kStages);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_step_kernel<kStages, false>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

template <int kStages, bool kPre>
cudaError_t set_smem_of() {
  cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<kStages, kPre>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(step_smem(kStages)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_step_kernel<kStages, kPre>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_step_kernel<kStages, kPre>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

// How many clusters of C fused-step CTAs the current device keeps resident
// at once (0 if the query fails). Needs set_step_smem() first.
int step_max_clusters(int C) { return max_clusters_of<kStStages>(C); }

cudaError_t set_step_smem() {
  const cudaError_t e = set_smem_of<kStStages, false>();
  return e != cudaSuccess ? e : set_smem_of<kStStages, true>();
}

cudaError_t launch_decode_step(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmpool,
                               const KvView& kv, int batch, const __nv_bfloat16* q, int hq, const msa_select_cfg& cfg,
                               int k_total, int C, int chunk, int bps, float scale_log2,
                               int32_t* idx_out, __nv_bfloat16* out, float* lse, int32_t* status,
                               const __nv_bfloat16* k, __nv_bfloat16* pooled_out, const float* pre_scores,
                               cudaStream_t stream) {
  StepArgs a;
  a.q = q;
  a.hq = hq;
  a.hkv = kv.hkv;
  a.grp = hq / kv.hkv;
  a.k_scored = cfg.k_scored;
  a.k_total = k_total;
  a.force_local = cfg.force_local;
  a.chunk = chunk;
  a.bps = bps;
  // sample keys per compute warp: the fewest that give the cluster at least
  // twice k_scored samples (their k-th largest bounds the selection from below)
  int p = 1;
  while (p < 8 && C * kStWarps * p < 2 * cfg.k_scored) p *= 2;
  a.samples_per_warp = p;
  a.scale_log2 = scale_log2;
  a.idx_out = idx_out;
  a.out = out;
  a.lse = lse;
  a.status = status;
  a.k = k;
  a.pooled_out = pooled_out;
  a.pre_scores = pre_scores;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(C, kv.hkv, batch);
  lc.blockDim = dim3(kStThreads, 1, 1);
  lc.dynamicSmemBytes = step_smem(kStStages);
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
  if (pre_scores != nullptr) return cudaLaunchKernelEx(&lc, decode_step_kernel<kStStages, true>, tmk, tmv, tmpool, kv, a);
  return cudaLaunchKernelEx(&lc, decode_step_kernel<kStStages, false>, tmk, tmv, tmpool, kv, a);
}

}  // namespace msa
