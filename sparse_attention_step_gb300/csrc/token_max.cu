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
// block maxima go to the score buffer that the fused decode step (or the
// top-k kernel) reads.
#include <float.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace msa {

namespace {

constexpr int kTmWarps = 4;
constexpr int kTmThreads = 32 * (kTmWarps + 1);
constexpr int kTmStages = 4;
constexpr int kTmStage = kBlock * kHeadDim * 2;  // 16 KB: one block of index keys
constexpr int kTmMaxChunk = 64;                  // candidate blocks per CTA, at most
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
  uint8_t* ring = smem_align1024(tm_raw);
  __shared__ uint64_t full[kTmStages], empty[kTmStages];
  __shared__ int32_t rowid[kTmMaxChunk];  // first index-key row of each block, -1 = bad page
  // The index queries are needed only until the scoring warps hold them in
  // registers, so the per-warp block maxima reuse their space (keeping three
  // CTAs' shared memory within one SM).
  __shared__ union {
    float qsum[kTmMaxHeads][kHeadDim];
    float part[kTmMaxChunk][kTmWarps][kTmMaxHeads];
  } sh;
  auto& qsum = sh.qsum;
  auto& part = sh.part;

  const int s = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (kv.layout == MSA_KV_CONTIGUOUS && warp == kTmWarps && lane == 0) {
    // While the kernel before this one finishes, the first blocks of this
    // chunk are pulled into L2 (a prefetch has no result: if that kernel
    // writes any of them, the loads, issued after it has completed, read its
    // values).
    const int64_t bp = static_cast<int64_t>(blockIdx.x) * a.chunk;
    for (int j = 0; j < kTmStages && bp + j < a.max_blocks; ++j) {
      const int32_t r = static_cast<int32_t>(static_cast<int64_t>(s) * kv.max_tokens + (bp + j) * kBlock);
      tma_prefetch_2d(&tmi, 0, r);
      tma_prefetch_2d(&tmi, 64, r);
    }
  }
  pdl_wait();
  const int64_t len = kv.seq_len(s, a.status, kIdScore);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  const int64_t nbf = len / kBlock;
  int64_t n_cand = (a.force_local & kForceLocal) ? min(nbf, nb - 1) : nbf;
  if (n_cand < 0) n_cand = 0;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * a.chunk;
  if (b0 >= n_cand) return;
  const int nblk = static_cast<int>(min(static_cast<int64_t>(a.chunk), n_cand - b0));

  // index-key row of candidate block j of this chunk (-1: bad page, never selected)
  auto row_of = [&](int j) -> int32_t {
    const int64_t b = b0 + j;
    if (kv.layout == MSA_KV_CONTIGUOUS) return static_cast<int32_t>(static_cast<int64_t>(s) * kv.max_tokens + b * kBlock);
    const int32_t p = kv.page(s, b, a.status, kIdScore);
    return p < 0 ? -1 : p * kBlock;
  };
  // The producer sets up the ring and issues the first stages at once, so
  // they are in flight while the index query is gathered.
  const int n_pre = min(kTmStages, nblk);
  if (warp == kTmWarps && lane == 0) {
    for (int i = 0; i < kTmStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kTmWarps);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmi);
    for (int j = 0; j < n_pre; ++j) {
      const int32_t r = row_of(j);
      uint8_t* dst = ring + j * kTmStage;
      mbar_arrive_expect_tx(&full[j], kTmStage);
      tma_load_2d(dst, &tmi, 0, r < 0 ? 0 : r, &full[j]);
      tma_load_2d(dst + kTmStage / 2, &tmi, 64, r < 0 ? 0 : r, &full[j]);
    }
  }
  if (tid < kTmMaxChunk) rowid[tid] = tid < nblk ? row_of(tid) : -1;
  if (tid < kTmMaxHeads * 16) {
    // group h's index query, dims [8e, 8e + 8): the group's query heads are
    // loaded at once (16 bytes each), then summed in head order
    const int hh = tid >> 4, e = tid & 15;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (hh < a.hkv) {
      const uint4* qg = reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(s) * a.hq + hh * a.grp) * kHeadDim) + e;
      uint4 x[kMaxGroupHeads];
#pragma unroll
      for (int g = 0; g < kMaxGroupHeads; ++g) x[g] = g < a.grp ? qg[g * (kHeadDim / 8)] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int g = 0; g < kMaxGroupHeads; ++g) {
        const uint32_t w[4] = {x[g].x, x[g].y, x[g].z, x[g].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] += __uint_as_float(w[i] << 16);
          acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) qsum[hh][8 * e + i] = acc[i];
  }
  __syncthreads();

  if (warp == kTmWarps) {
    if (lane == 0) {
      int issued = n_pre;
      for (int j = n_pre; j < nblk; ++j) {
        const int slot = j % kTmStages;
        if (j >= kTmStages && !mbar_wait(&empty[slot], ((j / kTmStages) - 1) & 1, a.status, kIdScore)) break;
        const int32_t y = rowid[j] < 0 ? 0 : rowid[j];
        uint8_t* dst = ring + slot * kTmStage;
        mbar_arrive_expect_tx(&full[slot], kTmStage);
        tma_load_2d(dst, &tmi, 0, y, &full[slot]);
        tma_load_2d(dst + kTmStage / 2, &tmi, 64, y, &full[slot]);
        issued = j + 1;
      }
      mbar_drain(full, kTmStages, issued, a.status, kIdScore);
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
    bar_sync_warps(1, 32 * kTmWarps);  // every scoring warp has read qsum: part may overwrite it
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
// tiles of a chunk batch, on the 5th-generation tensor cores. A CTA takes a
// chunk of index-key blocks of one sequence and a group of up to 16 of its
// tiles, for every KV head: the 128 index queries (tile x head) are the rows
// of A, the 128 index-key tokens of a pair of blocks the columns of B, so
//   D[query, token] = q_idx . K_idx[token]     tcgen05.mma M128 N128, fp32 in TMEM
// with the fp32 index queries split into a bf16 head (k-steps 0-7) and a bf16
// remainder (k-steps 8-15) accumulated into the same D, which reproduces the
// fp32 products to ~2^-16 relative (rows of absent tiles or heads are zeros).
// Each query row sits in one TMEM lane, so the maximum over a block's 64
// tokens is a reduction inside one thread. Warps: 0-3 read D (TMEM lanes
// 0-127), 4 the TMA producer (4-stage ring of block pairs), 5 the TMEM
// allocator and MMA issuer; D is double-buffered. The index queries come from
// the workspace (the prefill index-query kernel). grid (block chunks, groups
// of 16 tiles of one sequence), the chunk sized so the grid is about one wave.
// ---------------------------------------------------------------------------
namespace {
constexpr int kTpTiles = 16;       // tiles per group (x 8 heads = the MMA's 128 rows)
constexpr int kTpMaxChunk = 128;   // index-key blocks per CTA, at most (an even count)
constexpr int kTpThreads = 192;
constexpr int kTpProducer = 4, kTpMma = 5;  // warps
constexpr int kTpStages = 4;
// A stage holds a pair of blocks as the 128 rows of B: [block 2p, dims 0-63 |
// block 2p + 1, dims 0-63 | block 2p, dims 64-127 | block 2p + 1, dims 64-127],
// 8 KB each (64 rows of 128 bytes, 128-byte swizzle)
constexpr int kTpStage = 2 * kTmStage;
constexpr int kTpABytes = 65536;   // A: head and remainder, 128 rows x 128 dims bf16 each
struct TpTail {
  uint64_t kv_full[kTpStages];
  uint64_t kv_empty[kTpStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t rowid[kTpMaxChunk];
};
constexpr size_t kTpSmem = 1024 + kTpABytes + static_cast<size_t>(kTpStages) * kTpStage + sizeof(TpTail);
}  // namespace

struct TokenMaxPrefillArgs {
  const float* qidx;  // [tiles, hkv, 128] fp32
  int hkv;
  int chunk;  // index-key blocks per CTA: even, <= kTpMaxChunk
  int64_t max_blocks;
  float* scores;  // [tiles, hkv, max_blocks]
  int32_t* status;
};

__global__ void __launch_bounds__(kTpThreads, 1) token_max_prefill_kernel(const __grid_constant__ CUtensorMap tmi,
                                                                        KvView kv, TokenMaxPrefillArgs a,
                                                                        const PrefillBatch pb) {
  extern __shared__ __align__(1024) uint8_t tp_raw[];
  uint8_t* base = smem_align1024(tp_raw);
  uint8_t* qa = base;                  // A operands, 128-byte swizzled, K-major
  uint8_t* ring = base + kTpABytes;    // index-key block pairs
  TpTail& st = *reinterpret_cast<TpTail*>(ring + kTpStages * kTpStage);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the group's sequence: groups are counted sequence by sequence
  int seq = 0, first = 0;
  for (int sq = 0; sq < pb.n_seqs; ++sq) {
    const int n_g = (pb.tile_off[sq + 1] - pb.tile_off[sq] + kTpTiles - 1) / kTpTiles;
    seq = sq;
    if (static_cast<int>(blockIdx.y) < first + n_g) break;
    first += n_g;
  }
  const int j0 = (static_cast<int>(blockIdx.y) - first) * kTpTiles;  // first tile of the group within its sequence
  const int t0 = pb.tile_off[seq] + j0;                          // its global tile
  const int t_end = min(t0 + kTpTiles, pb.tile_off[seq + 1]);
  const int64_t diag0 = pb.q_start[seq] / kBlock + j0;           // candidates of tile t0 + t: blocks < diag0 + t
  const int64_t n_max = diag0 + (t_end - t0) - 1;                // the group's most candidates
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * a.chunk;
  if (b0 >= n_max) return;  // the whole CTA leaves before any barrier or allocation
  const int nblk = static_cast<int>(min(static_cast<int64_t>(a.chunk), n_max - b0));
  const int npair = (nblk + 1) / 2;
  pdl_wait();

  // index-key row of block j of this chunk, -1 for a bad page
  auto row_of = [&](int j) -> int32_t {
    const int64_t b = b0 + j;
    if (kv.layout == MSA_KV_CONTIGUOUS) return static_cast<int32_t>(static_cast<int64_t>(seq) * kv.max_tokens + b * kBlock);
    const int32_t p = kv.page(seq, b, a.status, kIdScore);
    return p < 0 ? -1 : p * kBlock;
  };
  auto issue_pair = [&](int p, int slot) {  // the producer: block pair p into ring slot `slot`
    const int nb_p = min(2, nblk - 2 * p);  // the last pair of an odd chunk has one block
    uint8_t* dst = ring + slot * kTpStage;
    mbar_arrive_expect_tx(&st.kv_full[slot], nb_p * kTmStage);
    for (int e = 0; e < nb_p; ++e) {
      const int32_t r = row_of(2 * p + e);
      const int32_t y = r < 0 ? 0 : r;
      tma_load_2d(dst + e * 8192, &tmi, 0, y, &st.kv_full[slot]);
      tma_load_2d(dst + 16384 + e * 8192, &tmi, 64, y, &st.kv_full[slot]);
    }
  };
  // The producer sets up the barriers and issues the first pairs at once, so
  // they travel while A is built.
  const int n_pre = min(kTpStages, npair);
  if (warp == kTpProducer && lane == 0) {
    for (int i = 0; i < kTpStages; ++i) {
      mbar_init(&st.kv_full[i], 1);
      mbar_init(&st.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&st.s_full[i], 1);
      mbar_init(&st.s_empty[i], 4);
    }
    mbar_init(&st.drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmi);
    for (int p = 0; p < n_pre; ++p) issue_pair(p, p);
  }
  if (tid < kTpMaxChunk) st.rowid[tid] = tid < nblk ? row_of(tid) : -1;
  // A: row r = 8 (tile) + head; 16-byte piece c16 of a row's 256 bytes goes to
  // [operand][dim half][row][(c16 mod 8) ^ (row mod 8)] (the TMA 128-byte swizzle).
  // Every index-query load of this thread is in flight before the first is used.
  constexpr int kAIt = (128 * 16 + kTpThreads - 1) / kTpThreads;
  float4 qu[kAIt], qv[kAIt];
#pragma unroll
  for (int it = 0; it < kAIt; ++it) {
    const int i = tid + it * kTpThreads;
    const int row = i >> 4, c16 = i & 15;
    const int g = row >> 3, h = row & 7;
    qu[it] = qv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < 128 * 16 && h < a.hkv && t0 + g < t_end) {
      const float4* qi = reinterpret_cast<const float4*>(a.qidx + (static_cast<int64_t>(t0 + g) * a.hkv + h) * kHeadDim +
                                                         8 * c16);
      qu[it] = qi[0];
      qv[it] = qi[1];
    }
  }
#pragma unroll
  for (int it = 0; it < kAIt; ++it) {
    const int i = tid + it * kTpThreads;
    if (i >= 128 * 16) break;
    const int row = i >> 4, c16 = i & 15;
    const float x[8] = {qu[it].x, qu[it].y, qu[it].z, qu[it].w, qv[it].x, qv[it].y, qv[it].z, qv[it].w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float h0 = __bfloat162float(__float2bfloat16_rn(x[2 * e]));
      const float h1 = __bfloat162float(__float2bfloat16_rn(x[2 * e + 1]));
      hi[e] = pack_bf16(h0, h1);
      lo[e] = pack_bf16(x[2 * e] - h0, x[2 * e + 1] - h1);
    }
    const int off = (c16 >> 3) * 16384 + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(qa + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(qa + 32768 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  fence_proxy_async();  // the tensor core reads A through the async proxy
  if (warp == kTpMma) {
    tc::alloc(&st.tmem_base, 256);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = st.tmem_base;

  if (warp == kTpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = n_pre;
      for (int p = n_pre; p < npair; ++p) {
        const int slot = p % kTpStages;
        if (p >= kTpStages && !mbar_wait(&st.kv_empty[slot], ((p / kTpStages) - 1) & 1, a.status, kIdScore)) break;
        issue_pair(p, slot);
        issued = p + 1;
      }
      // every load this thread issued has landed before the CTA may exit
      for (int p = issued - kTpStages < 0 ? 0 : issued - kTpStages; p < issued; ++p)
        mbar_wait(&st.kv_full[p % kTpStages], (p / kTpStages) & 1, a.status, kIdScore);
    }
  } else if (warp == kTpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // N = 128: the pair's two blocks (in an odd chunk's last pair, rows
      // 64-127 of B are stale and the columns they produce are not read)
      constexpr uint32_t kId = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t a_addr = smem_u32(qa), r_addr = smem_u32(ring);
      for (int p = 0; p < npair; ++p) {
        const int slot = p % kTpStages, buf = p & 1;
        if (!mbar_wait(&st.kv_full[slot], (p / kTpStages) & 1, a.status, kIdScore)) break;
        if (p >= 2 && !mbar_wait(&st.s_empty[buf], ((p >> 1) - 1) & 1, a.status, kIdScore)) break;
        tc::fence_after();
        const uint32_t d = tmem + buf * 128;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int k8 = kk & 7;  // k-steps 8-15 repeat the dims with the remainder of the queries
          const uint64_t ad = tc::sdesc_sw128(a_addr + (kk >> 3) * 32768 + (k8 >> 2) * 16384 + (k8 & 3) * 32, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(r_addr + slot * kTpStage + (k8 >> 2) * 16384 + (k8 & 3) * 32, 16, 1024);
          tc::mma_ss(d, ad, bd, kId, kk > 0 ? 1u : 0u);
        }
        tc::commit(&st.kv_empty[slot]);
        tc::commit(&st.s_full[buf]);
      }
      tc::commit(&st.drain);
      mbar_wait(&st.drain, 0, a.status, kIdScore);  // nothing of ours is left in flight
    }
  } else {
    // ------------------------------------------------------------ block maxima (query rows 0-127)
    const int row = 32 * warp + lane;
    const int g = row >> 3, h = row & 7;
    const bool live = h < a.hkv && t0 + g < t_end;
    const int64_t n_cand = diag0 + g;  // this tile's candidates
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    float* out = a.scores + (static_cast<int64_t>(live ? t0 + g : 0) * a.hkv + h) * a.max_blocks;
    for (int p = 0; p < npair; ++p) {
      const int buf = p & 1;
      if (!mbar_wait_warp(&st.s_full[buf], (p >> 1) & 1, a.status, kIdScore)) break;
      tc::fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tc::ld64(tmem + lane_base + buf * 128, r0, r1);       // block 2p
      tc::ld64(tmem + lane_base + buf * 128 + 64, r2, r3);  // block 2p + 1
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&st.s_empty[buf]);
      float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        m0 = fmaxf(m0, fmaxf(__uint_as_float(r0[c]), __uint_as_float(r1[c])));
        m1 = fmaxf(m1, fmaxf(__uint_as_float(r2[c]), __uint_as_float(r3[c])));
      }
      const int j = 2 * p;
      const int64_t b = b0 + j;
      if (live && b < n_cand) out[b] = st.rowid[j] < 0 ? -INFINITY : m0;  // bad page: never selected
      if (live && j + 1 < nblk && b + 1 < n_cand) out[b + 1] = st.rowid[j + 1] < 0 ? -INFINITY : m1;
    }
  }
  pdl_trigger();
  tc::fence_before();
  __syncthreads();
  if (warp == kTpMma) {
    tc::fence_after();
    tc::dealloc(tmem, 256);
  }
}

size_t token_max_prefill_smem_bytes() { return kTpSmem; }

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
  int groups = 0;  // groups of kTpTiles tiles, sequence by sequence
  for (int s = 0; s < pb.n_seqs; ++s) groups += (pb.tile_off[s + 1] - pb.tile_off[s] + kTpTiles - 1) / kTpTiles;
  if (last <= 0 || groups == 0) return cudaSuccess;  // no candidates anywhere
  // about one wave: one CTA per SM, the groups sharing the SMs
  int num_sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t per_group = max(static_cast<int64_t>(1), static_cast<int64_t>(num_sms > 0 ? num_sms : 1) / groups);
  int64_t chunk = (last + per_group - 1) / per_group;
  chunk = (chunk + 1) / 2 * 2;
  chunk = chunk < 16 ? 16 : chunk > kTpMaxChunk ? kTpMaxChunk : chunk;
  a.chunk = static_cast<int>(chunk);
  const unsigned chunks = static_cast<unsigned>((last + chunk - 1) / chunk);
  token_max_prefill_kernel<<<dim3(chunks, groups), kTpThreads, token_max_prefill_smem_bytes(), stream>>>(tmi, kv, a,
                                                                                                          pb);
  return cudaGetLastError();
}

size_t token_max_smem_bytes() { return 1024 + static_cast<size_t>(kTmStages) * kTmStage; }

cudaError_t set_token_max_smem() {
  cudaError_t e = cudaFuncSetAttribute(token_max_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(token_max_smem_bytes()));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(token_max_score_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
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
  // one wave: the batch's blocks spread evenly over the CTAs the device keeps
  // resident at once (its SMs x the CTAs that fit one SM, asked of the runtime)
  int num_sms = 0, dev = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, token_max_score_kernel, kTmThreads,
                                                    token_max_smem_bytes()) != cudaSuccess)
    return cudaGetLastError();
  const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * (per_sm > 0 ? per_sm : 1);
  int64_t chunk = (static_cast<int64_t>(batch) * a.max_blocks + slots - 1) / slots;
  chunk = chunk < 8 ? 8 : chunk > kTmMaxChunk ? kTmMaxChunk : chunk;
  a.chunk = static_cast<int>(chunk);
  const unsigned chunks = static_cast<unsigned>((a.max_blocks + chunk - 1) / chunk);
  // programmatic dependent launch: the CTAs may be placed while the previous
  // kernel drains; they wait for it before reading anything
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(chunks, batch, 1);
  lc.blockDim = dim3(kTmThreads, 1, 1);
  lc.dynamicSmemBytes = token_max_smem_bytes();
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, token_max_score_kernel, tmi, kv, a);
}

}  // namespace msa
