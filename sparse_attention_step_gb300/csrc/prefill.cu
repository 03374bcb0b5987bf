// Step 2, chunked prefill: causal softmax attention of a 64-token query tile's
// rows (tokens x group heads) over the blocks selected for that tile and KV
// head ("MiniMax goes sparse", §1 Step 2, and §3: in prefill the savings fall
// on the main attention).
//
// Rows of a unit (tile j, KV head h) are ordered token-major, head-minor:
// row r = t * G + gh is query token 64 j + t, head h * G + gh. A CTA owns 128
// rows (8 warps x 16 rows) and loops over the unit's blocks; a producer warp
// streams each 64x128 K/V block into a shared-memory ring with 2-D TMA copies
// (128-byte swizzle). Per block and warp: S = Q K^T (mma m16n8k16, bf16 in,
// fp32 accumulate), causal mask on the diagonal block, online softmax in fp32
// (exp2), O += P V with P taken straight from the S accumulators.
#include <float.h>

#include "kernels.cuh"

namespace msa {

constexpr int kPfWarps = 8;
constexpr int kPfThreads = 32 * (kPfWarps + 1);
constexpr int kPfRows = 16 * kPfWarps;  // rows per CTA
constexpr int kPfStageBytes = 4 * 8192;
constexpr int kPfStages = 4;
constexpr int kPfMaxList = 512;  // list entries per (tile, head); larger k_total is rejected on the host


struct PrefillSmemTail {
  uint64_t full[kPfStages];
  uint64_t empty[kPfStages];
  int32_t blocks[kPfMaxList];
  int32_t n_blocks;
};

// grid (row groups of 128, Hkv, n_tiles)
__global__ void __launch_bounds__(kPfThreads) prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv, KvView kv,
                                                                 PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_align1024(smem_raw);
  PrefillSmemTail& st = *reinterpret_cast<PrefillSmemTail*>(ring + kPfStages * kPfStageBytes);

  const int rg = blockIdx.x, h = blockIdx.y, tile = blockIdx.z;  // tile: global over the batch
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = a.batch.seq_of_tile(tile);
  const int jt = tile - a.batch.tile_off[seq];  // tile within its sequence
  const int64_t q_start = a.batch.q_start[seq];
  const int64_t len = kv.seq_len(seq, a.status, kIdPrefill);
  const int64_t diag = q_start / kBlock + jt;

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
        if (keep && pos < kPfMaxList) st.blocks[pos] = b;
        n += __popc(ballot);
      }
      if (n > kPfMaxList) {  // more valid entries than the kernel holds
        if (lane == 0) set_status(a.status, MSA_ERR_UNSUPPORTED, kIdPrefill);
        n = kPfMaxList;
      }
    } else {
      n = static_cast<int>(diag + 1);  // every causal block (list not materialised)
    }
    if (lane == 0) {
      st.n_blocks = n;
      for (int i = 0; i < kPfStages; ++i) {
        mbar_init(&st.full[i], 1);
        mbar_init(&st.empty[i], kPfWarps);
      }
      fence_mbar_init();
    }
  }
  __syncthreads();
  const int nblk = st.n_blocks;
  const bool dense = a.idx == nullptr;

  const int g = lane >> 2, c = lane & 3;
  if (warp == kPfWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        const int stg = i % kPfStages;
        if (i >= kPfStages && !mbar_wait(&st.empty[stg], ((i / kPfStages) - 1) & 1, a.status, kIdPrefill)) break;
        issued = i + 1;
        const int b = dense ? i : st.blocks[i];
        const int64_t row = kv.block_row(seq, h, b, a.status, kIdPrefill);
        uint8_t* dst = ring + stg * kPfStageBytes;
        mbar_arrive_expect_tx(&st.full[stg], kPfStageBytes);
        const int32_t y = static_cast<int32_t>(row < 0 ? 0 : row);
        tma_load_2d(dst, &tmk, 0, y, &st.full[stg]);
        tma_load_2d(dst + 8192, &tmk, 64, y, &st.full[stg]);
        tma_load_2d(dst + 16384, &tmv, 0, y, &st.full[stg]);
        tma_load_2d(dst + 24576, &tmv, 64, y, &st.full[stg]);
      }
      mbar_drain(st.full, kPfStages, issued, a.status, kIdPrefill);
    }
    return;  // the producer takes no part in the epilogue
  }

  // ---------------- consumers ----------------
  // this thread's two rows: g and g + 8 of the warp's 16-row slab
  int64_t pos[2];
  bool live[2];
  int64_t qrow[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = rg * kPfRows + 16 * warp + g + 8 * hr;
    const int t = r / a.grp, gh = r % a.grp;
    const int64_t tq = a.batch.tile_row0(seq, tile) + t;  // query index within its sequence's chunk
    live[hr] = (t < kBlock) && tq >= 0 && (tq < a.batch.q_cnt[seq]);
    pos[hr] = q_start + tq;
    qrow[hr] = live[hr] ? (a.batch.q_off[seq] + tq) * a.hq + h * a.grp + gh : 0;
  }
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const __nv_bfloat16* r0 = a.q + qrow[0] * kHeadDim + 16 * kk + 2 * c;
    const __nv_bfloat16* r1 = a.q + qrow[1] * kHeadDim + 16 * kk + 2 * c;
    qa[kk][0] = live[0] ? *reinterpret_cast<const uint32_t*>(r0) : 0u;
    qa[kk][1] = live[1] ? *reinterpret_cast<const uint32_t*>(r1) : 0u;
    qa[kk][2] = live[0] ? *reinterpret_cast<const uint32_t*>(r0 + 8) : 0u;
    qa[kk][3] = live[1] ? *reinterpret_cast<const uint32_t*>(r1 + 8) : 0u;
  }
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  // ldmatrix lane roles
  const int kb_row = (lane & 7) + ((lane >> 4) & 1) * 8;  // key within the 16-key pair of n-tiles
  const int kb_chunk = (lane >> 3) & 1;                    // dim half of the k-step
  const int vb_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // key within the 16-key step
  const int vb_chunk = (lane >> 4) & 1;                    // dim n-tile of the pair

  for (int i = 0; i < nblk; ++i) {
    const int stg = i % kPfStages;
    if (!mbar_wait_warp(&st.full[stg], (i / kPfStages) & 1, a.status, kIdPrefill)) break;
    const int b = dense ? i : st.blocks[i];
    const uint32_t kbase = smem_u32(ring + stg * kPfStageBytes);
    const uint32_t vbase = kbase + 16384;
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // pairs of key n-tiles
        uint32_t b0, b1, b2, b3;
        const int key = 16 * np + kb_row;
        ldsm_x4(kbase + (kk >> 2) * 8192 + swz128(key, (kk & 3) * 2 + kb_chunk), b0, b1, b2, b3);
        mma_bf16(sc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16(sc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }
    // mask and scale
    const int64_t key0 = static_cast<int64_t>(b) * kBlock;
    const bool need_mask = (key0 + kBlock - 1 > diag * kBlock) || (key0 + kBlock > len);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        float z = sc[nt][e] * a.scale_log2;
        if (need_mask || !live[hr]) {
          const int64_t kp = key0 + 8 * nt + 2 * c + (e & 1);
          if (!live[hr] || kp > pos[hr] || kp >= len) z = -INFINITY;
        }
        sc[nt][e] = z;
        mx[hr] = fmaxf(mx[hr], z);
      }
    }
    float al[2], ref[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float mn = fmaxf(m[hr], mx[hr]);
      ref[hr] = mn == -INFINITY ? 0.f : mn;
      al[hr] = exp2f(m[hr] - ref[hr]);
      m[hr] = mn;
      l[hr] *= al[hr];
    }
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      o[dt][0] *= al[0]; o[dt][1] *= al[0]; o[dt][2] *= al[1]; o[dt][3] *= al[1];
    }
    uint32_t pa[4][4];  // P as A fragments, one per 16-key step
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      float p[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = exp2f(sc[2 * ks][e] - ref[e >> 1]);
        p[4 + e] = exp2f(sc[2 * ks + 1][e] - ref[e >> 1]);
      }
      l[0] += p[0] + p[1] + p[4] + p[5];
      l[1] += p[2] + p[3] + p[6] + p[7];
      pa[ks][0] = pack_bf16(p[0], p[1]);  // row g,   keys 2c..
      pa[ks][1] = pack_bf16(p[2], p[3]);  // row g+8, keys 2c..
      pa[ks][2] = pack_bf16(p[4], p[5]);  // row g,   keys 8+2c..
      pa[ks][3] = pack_bf16(p[6], p[7]);  // row g+8, keys 8+2c..
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {  // pairs of dim n-tiles
        uint32_t b0, b1, b2, b3;
        const int key = 16 * ks + vb_row;
        ldsm_x4_t(vbase + (dp >> 2) * 8192 + swz128(key, (dp & 3) * 2 + vb_chunk), b0, b1, b2, b3);
        mma_bf16(o[2 * dp], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
        mma_bf16(o[2 * dp + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&st.empty[stg]);
  }
  // epilogue: finish the row sums across the 4 lanes of a row, normalise, store
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
    l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    if (!live[hr]) continue;
    const float inv = l[hr] > 0.f ? 1.f / l[hr] : 0.f;
    __nv_bfloat16* dst = a.out + qrow[hr] * kHeadDim + 2 * c;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      *reinterpret_cast<uint32_t*>(dst + 8 * dt) = pack_bf16(o[dt][2 * hr] * inv, o[dt][2 * hr + 1] * inv);
    }
    if (a.lse != nullptr && c == 0) a.lse[qrow[hr]] = l[hr] > 0.f ? m[hr] * kLn2 + logf(l[hr]) : -INFINITY;
  }
}

size_t prefill_smem_bytes() { return 1024 + kPfStages * kPfStageBytes + sizeof(PrefillSmemTail); }

cudaError_t set_prefill_smem() {
  return cudaFuncSetAttribute(prefill_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(prefill_smem_bytes()));
}

cudaError_t launch_prefill_bf16(const CUtensorMap& tmk, const CUtensorMap& tmv, const KvView& kv,
                                const PrefillArgs& a, cudaStream_t stream) {
  const int row_groups = (kBlock * a.grp + kPfRows - 1) / kPfRows;
  dim3 grid(row_groups, kv.hkv, a.batch.total_tiles());
  prefill_bf16_kernel<<<grid, kPfThreads, prefill_smem_bytes(), stream>>>(tmk, tmv, kv, a);
  return cudaGetLastError();
}

}  // namespace msa
