// Step 2, chunked prefill on the 5th-generation tensor cores ("MiniMax goes
// sparse", §1 Step 2: the heads of a group share one list of KV blocks, the
// set is staged on chip in one pass and attended with a flash-style kernel).
//
// One CTA owns 256 query rows of a (64-token tile, KV head) unit: 32 tokens x
// the 8 heads of the group, as two M = 128 tiles (rows token-major,
// head-minor). The selected blocks are taken two at a time (a pair of 128
// keys; an odd count ends with a single block). For every pair:
//   S_t = Q_t K^T      tcgen05.mma M128 N128 K16 x 8 (N64 for a single
//                      block), bf16 -> fp32 in TMEM
//   softmax            tcgen05.ld of the scores, causal mask on the diagonal
//                      block, online max with lazy rescaling (O is rescaled
//                      in TMEM only when the running max grows by more than
//                      2^8), exp2; P (bf16, two per 32-bit column) is stored
//                      back over the scores it came from
//   O_t += P_t V       tcgen05.mma M128 N128 K16 x 8 (x 4) with A = P read
//                      from TMEM and V read MN-major from shared memory
// An M128 MMA costs about the same at N = 64 as at N = 128, so scoring a pair
// at once halves the tensor time of Q K^T against one block at a time.
// Warp roles: warps 0-7 softmax of tile 0 and warps 8-15 of tile 1; within a
// tile, warp w takes 16 rows of the TMEM lanes 32 (w mod 4) .. (a warp
// reaches only those lanes), both halves of each: its threads j < 16 hold the
// pair's first block (score columns 0-63) and threads j + 16 the second
// (columns 64-127) of the same row (the 16x32bx2 TMEM access shape), so the
// halves exchange their maxima and sums with a shuffle. Warp 16 is
// the TMA producer (Q once, then 2-stage K and V rings of one pair each; K of
// a stage is released once both tiles' S are computed, V once both tiles'
// O += P V are), warp 17 the TMEM allocator and MMA issuer. The two tiles
// ping-pong: the tensor core runs one tile's MMAs while the other tile's
// softmax runs; the tensor core executes in issue order, so S of the next
// pair, issued after O += P V of this one, never overwrites a P still to be
// read, and once it has completed O of the tile is quiet for the softmax to
// rescale. TMEM: S / P of tile t in [128 t, 128 t + 128), O_t in
// [256 + 128 t, 384 + 128 t).
#include <float.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace msa {

namespace {

constexpr int kTcTiles = 2;
constexpr int kTcStages = 2;        // K and V rings, one pair of blocks per stage
constexpr int kPairBytes = 32768;   // two blocks x 64 rows x 128 dims of K (or V), bf16
constexpr int kSoftmaxWarps = 16;
constexpr int kTcThreads = 32 * (kSoftmaxWarps + 2);
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr uint32_t kTmemCols = 512;
constexpr int kQBytes = kTcTiles * 2 * 16384;   // two tiles x two 64-dim halves
constexpr int kRingBytes = kTcStages * kPairBytes;
constexpr int kMaxList = 512;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)

struct TcTail {
  uint64_t q_full;
  uint64_t k_full[kTcStages];
  uint64_t k_empty[kTcStages];
  uint64_t v_full[kTcStages];
  uint64_t v_empty[kTcStages];
  uint64_t s_full[kTcTiles];
  uint64_t p_full[kTcTiles];
  uint64_t o_final[kTcTiles];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t n_blocks;
  int32_t abort;
  int32_t blocks[kMaxList];
};

constexpr size_t kTcSmem = 1024 + kQBytes + 2 * kRingBytes + sizeof(TcTail);

__device__ inline float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Paired fp32 arithmetic (one instruction for two lanes of a float2).
__device__ inline float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 pa, pb, pc, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n mov.b64 pc, {%6, %7};\n"
      " fma.rn.f32x2 pd, pa, pb, pc;\n mov.b64 {%0, %1}, pd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ inline float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n add.rn.f32x2 pd, pa, pb;\n"
      " mov.b64 {%0, %1}, pd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ inline float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ inline void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ inline bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int32_t* abort, int32_t* status) {
  if (*abort) return false;
  if (!mbar_wait(bar, parity, status, kIdPrefill)) {
    *abort = 1;
    return false;
  }
  return true;
}

}  // namespace

// grid (2 row halves, Hkv, n_tiles); requires G = 8.
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                                                                  const __grid_constant__ CUtensorMap tmk,
                                                                  const __grid_constant__ CUtensorMap tmv, KvView kv,
                                                                  PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_align1024(smem_raw);
  uint8_t* qs = base;
  uint8_t* ks = base + kQBytes;            // K ring: [stage][dim half][128 keys][128 B]
  uint8_t* vs = ks + kRingBytes;           // V ring, the same layout
  TcTail& st = *reinterpret_cast<TcTail*>(vs + kRingBytes);

  const int rh = blockIdx.x, h = blockIdx.y, tile = blockIdx.z;  // tile: global over the batch
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = a.batch.seq_of_tile(tile);
  const int jt = tile - a.batch.tile_off[seq];  // tile within its sequence
  const int64_t diag = a.batch.q_start[seq] / kBlock + jt;

  if (warp == kProducerWarp && lane == 0) {
    mbar_init(&st.q_full, 1);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&st.k_full[i], 1);
      mbar_init(&st.k_empty[i], 1);
      mbar_init(&st.v_full[i], 1);
      mbar_init(&st.v_empty[i], 1);
    }
    for (int t = 0; t < kTcTiles; ++t) {
      mbar_init(&st.s_full[t], 1);
      mbar_init(&st.p_full[t], kSoftmaxWarps / 2);
      mbar_init(&st.o_final[t], 1);
    }
    mbar_init(&st.drain, 1);
    fence_mbar_init();
    // Q needs nothing of the list: its load starts while the list is read
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    mbar_arrive_expect_tx(&st.q_full, kQBytes);
    // first token of the row half (may be before the chunk, then the load
    // reads the fill value or another sequence's rows, never used)
    const int32_t tok0 = a.batch.q_off[seq] + a.batch.tile_row0(seq, tile) + rh * (kTcTiles * 16);
    for (int t = 0; t < kTcTiles; ++t)
      for (int half = 0; half < 2; ++half)
        tma_load_3d(qs + t * 32768 + half * 16384, &tmq, 64 * half, h * 8, tok0 + 16 * t, &st.q_full);
  }
  if (warp == 0) {
    // the valid entries of the unit's list, in order, read 32 at a time
    int n = 0;
    if (a.idx != nullptr) {
      const int32_t* list = a.idx + (static_cast<int64_t>(tile) * a.hkv + h) * a.k_total;
      for (int base = 0; base < a.k_total; base += 32) {
        const int32_t b = base + lane < a.k_total ? list[base + lane] : -1;
        if (b > diag) set_status(a.status, MSA_ERR_DEVICE_BOUNDS, kIdPrefill);
        const bool keep = b >= 0 && b <= diag;
        const uint32_t ballot = __ballot_sync(0xffffffffu, keep);
        const int pos = n + __popc(ballot & ((1u << lane) - 1u));
        if (keep && pos < kMaxList) st.blocks[pos] = b;
        n += __popc(ballot);
      }
      if (n > kMaxList) {  // more valid entries than the kernel holds
        if (lane == 0) set_status(a.status, MSA_ERR_UNSUPPORTED, kIdPrefill);
        n = kMaxList;
      }
    } else {
      n = static_cast<int>(diag + 1);
    }
    if (lane == 0) {
      st.n_blocks = n;
      st.abort = 0;
    }
  }
  if (warp == kMmaWarp) {
    tc::alloc(&st.tmem_base, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const int nblk = st.n_blocks;
  const int npair = (nblk + 1) >> 1;
  const bool dense = a.idx == nullptr;
  const uint32_t tmem = st.tmem_base;
  volatile int32_t* abort = &st.abort;
  auto blocks_in = [&](int i) { return nblk - 2 * i >= 2 ? 2 : 1; };  // blocks in pair i

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued_k = 0, issued_v = 0;
      for (int i = 0; i < npair; ++i) {
        const int stg = i % kTcStages, use = i / kTcStages, nb = blocks_in(i);
        auto row_of = [&](int j) {
          const int b = dense ? 2 * i + j : st.blocks[2 * i + j];
          const int64_t row = kv.block_row(seq, h, b, a.status, kIdPrefill);
          return static_cast<int32_t>(row < 0 ? 0 : row);
        };
        const int32_t y0 = row_of(0), y1 = nb == 2 ? row_of(1) : 0;
        // block j of the pair: rows [64 j, 64 j + 64) of each 64-dim half
        if (i >= kTcStages && !wait_or_abort(&st.k_empty[stg], (use - 1) & 1, abort, a.status)) break;
        mbar_arrive_expect_tx(&st.k_full[stg], nb * 16384);
        for (int j = 0; j < nb; ++j)
          for (int hd = 0; hd < 2; ++hd)
            tma_load_2d(ks + stg * kPairBytes + hd * 16384 + j * 8192, &tmk, 64 * hd, j ? y1 : y0, &st.k_full[stg]);
        issued_k = i + 1;
        if (i >= kTcStages && !wait_or_abort(&st.v_empty[stg], (use - 1) & 1, abort, a.status)) break;
        mbar_arrive_expect_tx(&st.v_full[stg], nb * 16384);
        for (int j = 0; j < nb; ++j)
          for (int hd = 0; hd < 2; ++hd)
            tma_load_2d(vs + stg * kPairBytes + hd * 16384 + j * 8192, &tmv, 64 * hd, j ? y1 : y0, &st.v_full[stg]);
        issued_v = i + 1;
      }
      // The CTA that starts when this one ends is, in the dispatch order, one
      // wave (a CTA per SM) later: its Q and first pair of K/V blocks are
      // pulled into L2 now, while this CTA's last pairs compute, so its
      // set-up does not wait on HBM. (Only a prefetch: nothing depends on the
      // guess.)
      {
        const int64_t nx = static_cast<int64_t>(blockIdx.x) + gridDim.x * (blockIdx.y + static_cast<int64_t>(gridDim.y) * blockIdx.z) +
                           a.num_sms;
        if (nx < static_cast<int64_t>(gridDim.x) * gridDim.y * gridDim.z) {
          const int rh2 = static_cast<int>(nx % gridDim.x), h2 = static_cast<int>((nx / gridDim.x) % gridDim.y);
          const int tile2 = static_cast<int>(nx / (static_cast<int64_t>(gridDim.x) * gridDim.y));
          const int seq2 = a.batch.seq_of_tile(tile2);
          const int64_t diag2 = a.batch.q_start[seq2] / kBlock + (tile2 - a.batch.tile_off[seq2]);
          const int32_t tok2 = a.batch.q_off[seq2] + a.batch.tile_row0(seq2, tile2) + rh2 * (kTcTiles * 16);
          for (int t = 0; t < kTcTiles; ++t)
            for (int half = 0; half < 2; ++half) tma_prefetch_3d(&tmq, 64 * half, h2 * 8, tok2 + 16 * t);
          const int n_first = a.idx == nullptr ? 2 : min(2, a.k_total);  // the dense list is 0 .. diag
          for (int j = 0; j < n_first; ++j) {
            const int32_t b = a.idx == nullptr ? j : a.idx[(static_cast<int64_t>(tile2) * a.hkv + h2) * a.k_total + j];
            if (b < 0 || b > diag2) continue;
            if (kv.layout != MSA_KV_CONTIGUOUS) continue;  // paged: the page lookup is left to the CTA itself
            const int32_t y = static_cast<int32_t>(kv.block_row(seq2, h2, b, nullptr, kIdPrefill));
            for (int hd = 0; hd < 2; ++hd) {
              tma_prefetch_2d(&tmk, 64 * hd, y);
              tma_prefetch_2d(&tmv, 64 * hd, y);
            }
          }
        }
      }
      // drain: every load this thread issued has landed before the CTA may exit
      mbar_wait(&st.q_full, 0, a.status, kIdPrefill);
      for (int i = issued_k - kTcStages < 0 ? 0 : issued_k - kTcStages; i < issued_k; ++i)
        mbar_wait(&st.k_full[i % kTcStages], (i / kTcStages) & 1, a.status, kIdPrefill);
      for (int i = issued_v - kTcStages < 0 ? 0 : issued_v - kTcStages; i < issued_v; ++i)
        mbar_wait(&st.v_full[i % kTcStages], (i / kTcStages) & 1, a.status, kIdPrefill);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS2 = tc::idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t kIdS1 = tc::idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t kIdO = tc::idesc_bf16(128, 128, 0, 1);
      const uint32_t q_addr = smem_u32(qs), k_addr = smem_u32(ks), v_addr = smem_u32(vs);
      // S_t = Q_t K^T over the pair's keys (K-major, 128 B rows, 8-row groups 1 KB apart)
      auto issue_s = [&](int t, int i) {
        const uint32_t d = tmem + t * 128;
        const uint32_t id = blocks_in(i) == 2 ? kIdS2 : kIdS1;
        const uint32_t kb = k_addr + (i % kTcStages) * kPairBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t ad = tc::sdesc_sw128(q_addr + t * 32768 + off, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(kb + off, 16, 1024);
          tc::mma_ss(d, ad, bd, id, kk > 0);
        }
      };
      // O_t += P V with P (bf16, packed in pairs) over the scores of the pair;
      // V MN-major: 16 keys a step, the two 64-dim halves 16 KB apart
      auto issue_pv = [&](int t, int i) {
        const uint32_t d = tmem + 256 + t * 128;
        const uint32_t vb = v_addr + (i % kTcStages) * kPairBytes;
        const int steps = 4 * blocks_in(i);
        for (int s = 0; s < steps; ++s) {
          const uint64_t bd = tc::sdesc_sw128(vb + s * 2048, 16384, 1024);
          tc::mma_ts(d, tmem + t * 128 + 8 * s, bd, kIdO, (i > 0 || s > 0) ? 1u : 0u);
        }
      };
      bool ok = wait_or_abort(&st.q_full, 0, abort, a.status);
      tc::fence_after();
      if (ok && npair > 0 && (ok = wait_or_abort(&st.k_full[0], 0, abort, a.status))) {
        tc::fence_after();
        for (int t = 0; t < kTcTiles; ++t) {
          issue_s(t, 0);
          tc::commit(&st.s_full[t]);
        }
        tc::commit(&st.k_empty[0]);  // the K stage is free once both tiles' S have completed
      }
      // tensor-core order per pair i: O_0 += P_0 V, S_0 of pair i + 1,
      // O_1 += P_1 V, S_1 of pair i + 1
      for (int i = 0; ok && i < npair; ++i) {
        const int stg = i % kTcStages;
        const bool next = i + 1 < npair;
        if (!(ok = wait_or_abort(&st.v_full[stg], (i / kTcStages) & 1, abort, a.status))) break;
        if (!(ok = wait_or_abort(&st.p_full[0], i & 1, abort, a.status))) break;
        tc::fence_after();
        issue_pv(0, i);
        if (next) {
          if (!(ok = wait_or_abort(&st.k_full[(i + 1) % kTcStages], ((i + 1) / kTcStages) & 1, abort, a.status)))
            break;
          tc::fence_after();
          issue_s(0, i + 1);
          tc::commit(&st.s_full[0]);
        }
        if (!(ok = wait_or_abort(&st.p_full[1], i & 1, abort, a.status))) break;
        tc::fence_after();
        issue_pv(1, i);
        tc::commit(&st.v_empty[stg]);
        if (next) {
          issue_s(1, i + 1);
          tc::commit(&st.s_full[1]);
          tc::commit(&st.k_empty[(i + 1) % kTcStages]);
        }
      }
      for (int t = 0; t < kTcTiles; ++t) tc::commit(&st.o_final[t]);
      tc::commit(&st.drain);
      mbar_wait(&st.drain, 0, a.status, kIdPrefill);  // nothing of ours is left in flight
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Each warp takes 16 rows of its TMEM lane quadrant, both halves of each
    // row: thread j < 16 the scores of the pair's first block (columns
    // [0, 64)), thread j + 16 those of the second (columns [64, 128)) of the
    // same row, so the two halves meet by a shuffle.
    const int t = warp >> 3;                // tile
    const int q4 = warp & 3;                // TMEM lane quadrant (the lanes this warp may access)
    const int sub = (warp >> 2) & 1;        // its lanes [16 sub, 16 sub + 16) of the quadrant
    const int hf = lane >> 4;               // block of the pair: score columns [64 hf, 64 hf + 64)
    const int r = 32 * q4 + 16 * sub + (lane & 15);  // row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4 + 16 * sub) << 16;
    const int bar_id = 1 + t;               // the tile's 8 softmax warps
    const int tt = rh * (kTcTiles * 16) + 16 * t + (r >> 3);  // token within the 64-token tile
    const int head = h * 8 + (r & 7);
    const int64_t tl = a.batch.tile_row0(seq, tile) + tt;  // token within its sequence's chunk
    const bool live = tl >= 0 && tl < a.batch.q_cnt[seq];
    const int64_t tq = a.batch.q_off[seq] + tl;                 // its row in q and out
    float m = -INFINITY, l = 0.f;  // running max (log2 units) and this half's running sum
    bool ok = true;
    // Every warp of the tile runs every iteration and every named barrier, even
    // after a wait gave up (then it skips the work), so no partner warp can be
    // left waiting at a barrier.
    for (int i = 0; i < npair; ++i) {
      ok = __all_sync(0xffffffffu, ok && wait_or_abort(&st.s_full[t], i & 1, abort, a.status));
      tc::fence_after();
      const bool have = hf < blocks_in(i);  // the odd last pair has no second block
      uint32_t sa[32], sb[32];
      if (ok) {  // the whole warp loads (columns 64 hf .. 64 hf + 63 of its rows)
        tc::ld64_h2(tmem + lane_base + t * 128, sa, sb);
        tc::wait_ld();
      }
      if (!(ok && have)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sa[c] = sb[c] = __float_as_uint(-INFINITY);
      }
      const int b = !have ? -1 : dense ? 2 * i + hf : st.blocks[2 * i + hf];
      if (b == diag) {  // causal mask inside the diagonal block
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c > tt) sa[c] = __float_as_uint(-INFINITY);
          if (32 + c > tt) sb[c] = __float_as_uint(-INFINITY);
        }
      }
      float mx;
      {
        auto val = [&](int k) { return __uint_as_float(k < 32 ? sa[k] : sb[k - 32]); };
        float u[22], w[8];
#pragma unroll
        for (int k = 0; k < 21; ++k) u[k] = fmax3(val(3 * k), val(3 * k + 1), val(3 * k + 2));
        u[21] = val(63);
#pragma unroll
        for (int k = 0; k < 7; ++k) w[k] = fmax3(u[3 * k], u[3 * k + 1], u[3 * k + 2]);
        w[7] = u[21];
        mx = fmax3(fmax3(w[0], w[1], w[2]), fmax3(w[3], w[4], w[5]), fmaxf(w[6], w[7]));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the row's other half
      const float m_blk = mx * a.scale_log2;  // -inf stays -inf
      const float m_new = fmaxf(m, m_blk);
      const bool need = (m == -INFINITY) ? (m_new != -INFINITY) : (m_new > m + kRescaleLog2);
      // the rows of this warp (both halves of each are in it, so both take the
      // same decision) move to the new max together
      const bool resc = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (resc) {
        alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
        l *= alpha;
        m = m_new;
      }
      const float neg_ref = (m == -INFINITY) ? 0.f : -m;
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nr2 = make_float2(neg_ref, neg_ref);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
      // P replaces the scores it came from: columns [32 hf, 32 hf + 32) of the
      // tile's S buffer hold keys [64 hf, 64 hf + 64) in pairs (the row's
      // other half, in this warp, read those columns in the load above; no
      // other warp touches these rows). The next S into the buffer is issued
      // after O += P V of this pair.
      auto exp_store = [&](const uint32_t (&sr)[32], uint32_t col) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nr2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (c & 1) acc1 = fadd2(acc1, pp);
          else acc0 = fadd2(acc0, pp);
          pk[c] = pack_bf16(pp.x, pp.y);
        }
        // threads j < 16 store at `col`, threads j + 16 at `col` + 32 (for a
        // missing second block they store zeros, which nothing reads)
        if (ok) tc::st16_h2<32>(tmem + lane_base + t * 128 + col, pk);
      };
      exp_store(sa, 0);
      exp_store(sb, 16);
      const float2 acc = fadd2(acc0, acc1);
      const float sum = acc.x + acc.y;
      // O of this half rescaled to the new max (after the scores are consumed,
      // to keep the registers of both under the per-thread budget)
      if (resc && i > 0 && ok) {
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          const uint32_t oa = tmem + lane_base + 256 + t * 128 + cc * 32;  // columns + 64 hf
          tc::ld32_h2(oa, o);
          tc::wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tc::st32_h2<64>(oa, o);
        }
      }
      tc::wait_st();
      l += sum;
      tc::fence_before();
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&st.p_full[t]);
    }
    // epilogue: the row's two half sums, then O / l in bf16 and the lse
    const float L = l + __shfl_xor_sync(0xffffffffu, l, 16);
    ok = __all_sync(0xffffffffu, ok && wait_or_abort(&st.o_final[t], 0, abort, a.status));
    tc::fence_after();
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    // O / l in bf16 goes through the tile's half of the Q buffer (idle: every
    // MMA has completed), one 256-byte row per score row with its 16-byte
    // chunks XOR-swizzled by the row, so that the global stores below are
    // whole 512-byte runs instead of one 16-byte piece per row
    uint8_t* ob = qs + t * 32768;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t o[32];
      tc::ld32_h2(tmem + lane_base + 256 + t * 128 + cc * 32, o);  // columns + 64 hf
      tc::wait_ld();
      if (nblk == 0 || !ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint4 v;
        v.x = pack_bf16(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
        v.y = pack_bf16(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
        v.z = pack_bf16(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
        v.w = pack_bf16(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
        const int c = 8 * hf + 4 * cc + j / 8;  // 16-byte chunk of the row
        *reinterpret_cast<uint4*>(ob + r * 256 + ((c ^ (r & 7)) << 4)) = v;
      }
    }
    named_bar_sync(bar_id, 256);
    {
      // warp w of the tile stores tokens 2w and 2w + 1 of the tile: a token's
      // 8 heads are 2 KB contiguous in the output, 512 bytes per instruction
      const int wt = warp & 7;
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * wt + jj;
        const int64_t tlj = a.batch.tile_row0(seq, tile) + rh * (kTcTiles * 16) + 16 * t + j;
        if (tlj < 0 || tlj >= a.batch.q_cnt[seq]) continue;
        uint4* gdst = reinterpret_cast<uint4*>(a.out + ((a.batch.q_off[seq] + tlj) * a.hq + h * 8) * kHeadDim);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int qq = 32 * p + lane;  // 16-byte chunk of the token's 2 KB
          const int row = 8 * j + (qq >> 4), c = qq & 15;
          gdst[qq] = *reinterpret_cast<const uint4*>(ob + row * 256 + ((c ^ (row & 7)) << 4));
        }
      }
    }
    if (live && hf == 0 && a.lse != nullptr)
      a.lse[tq * a.hq + head] = (L > 0.f) ? (m * kLn2 + logf(L)) : -INFINITY;
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

size_t prefill_tc_smem_bytes() { return kTcSmem; }

cudaError_t set_prefill_tc_smem() {
  return cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kTcSmem));
}

cudaError_t launch_prefill_tc(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const KvView& kv, const PrefillArgs& a, cudaStream_t stream) {
  dim3 grid(2, kv.hkv, a.batch.total_tiles());
  PrefillArgs args = a;
  int dev = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&args.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) args.num_sms = 1;
  prefill_tc_kernel<<<grid, kTcThreads, kTcSmem, stream>>>(tmq, tmk, tmv, kv, args);
  return cudaGetLastError();
}

}  // namespace msa
