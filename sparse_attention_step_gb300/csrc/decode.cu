// Step 2, decode: softmax attention of the G query heads of a GQA group over
// the selected KV blocks of their group ("MiniMax goes sparse", §1 Step 2:
// the group loads one set of KV blocks and all its heads attend over it).
//
// One CTA handles a slice of one (sequence, KV head) unit's block list
// (split-K). bf16 path:
//   warp 4 (one lane) is the producer: it streams each selected 64x128 K and V
//     block into a ring of shared-memory stages with 2-D TMA copies (two
//     64-column boxes per tensor, 128-byte swizzle), one mbarrier per stage.
//   warps 0-3 are consumers: warp w owns tokens [16w, 16w+16) of every block.
//     S = K_w Q^T on tensor cores (mma m16n8k16: 16 tokens x 8 heads x 16
//     dims), online softmax per head in fp32 (exp2 with log2(e) folded into
//     the scale), then O^T += V_w^T P^T (16 dims x 8 heads x 16 tokens); P^T
//     comes from the S accumulators by an 8x8 transpose (movmatrix).
// The four warps' (m, l, O) are merged in shared memory; with several splits
// each CTA writes its partial to the workspace and the last CTA of the unit to
// finish (atomic ticket) merges them:
//   m = max_i m_i, l = sum_i l_i 2^(m_i - m), o = sum_i o_i 2^(m_i - m) / l.
// No CTA ever waits for another one.
//
// fp32 KV path: the same split/merge structure with a CUDA-core consumer
// (warp per 16 tokens, lane per 4 dims); used for fp32 caches only.
#include <float.h>

#include "kernels.cuh"

namespace msa {

constexpr int kMaxGroup = 8;           // query heads per KV head handled per CTA
constexpr int kDecConsumers = 4;       // consumer warps
constexpr int kDecThreads = 32 * (kDecConsumers + 1);
constexpr int kStageBytes = 4 * 8192;  // K (2 x 64x64 bf16) + V (2 x 64x64 bf16)
constexpr int kMaxListPerCta = 512;    // selected blocks handled by one CTA
constexpr int kPartFloats = 2 * kMaxGroup + kMaxGroup * kHeadDim;  // m[8], l[8], o[8][128]
constexpr int kOStride = kHeadDim + 4;  // padded row of the merge buffer
constexpr int kMaxSplits = 256;         // CTAs per unit (split-K)


// Shared memory of one CTA (after the 1024-aligned stage ring).
struct DecodeSmemTail {
  uint64_t full[8];
  uint64_t empty[8];
  int32_t blocks[kMaxListPerCta];
  int32_t n_blocks;
  int32_t dense_lo;  // dense: block i of this CTA is dense_lo + i (no list)
  int32_t is_last;
  float wm[kDecConsumers][kMaxGroup];
  float wl[kDecConsumers][kMaxGroup];
};

// Writes the per-warp state into the merge buffer (rows = heads, padded).
// Then merges `nw` states -> (M, L, O) for head/dims owned by this thread.
__device__ inline void merge_states(int nw, const float* wm, const float* wl, int wstride, const float* o,
                                    int ostride_w, int head, int d0, float& M, float& L, float (&acc)[8]) {
  M = -INFINITY;
  for (int w = 0; w < nw; ++w) M = fmaxf(M, wm[w * wstride + head]);
  L = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (M == -INFINITY) return;
  for (int w = 0; w < nw; ++w) {
    const float f = exp2f(wm[w * wstride + head] - M);
    L += f * wl[w * wstride + head];
    const float* src = o + w * ostride_w + head * kOStride + d0;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(f, src[i], acc[i]);
  }
}

template <typename T>
__device__ inline void store_out8(T* dst, const float (&x)[8]);
template <>
__device__ inline void store_out8<__nv_bfloat16>(__nv_bfloat16* dst, const float (&x)[8]) {
  uint4 o;
  o.x = pack_bf16(x[0], x[1]);
  o.y = pack_bf16(x[2], x[3]);
  o.z = pack_bf16(x[4], x[5]);
  o.w = pack_bf16(x[6], x[7]);
  *reinterpret_cast<uint4*>(dst) = o;
}
template <>
__device__ inline void store_out8<float>(float* dst, const float (&x)[8]) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// Final normalisation of one (head, 8 dims) piece.
template <typename T>
__device__ inline void write_final(const DecodeArgs& a, int s, int h, int head, int d0, float M, float L,
                                   const float (&acc)[8]) {
  float x[8];
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = acc[i] * inv;
  const int64_t qrow = static_cast<int64_t>(s) * a.hq + h * a.grp + head;
  store_out8<T>(reinterpret_cast<T*>(a.out) + qrow * kHeadDim + d0, x);
  if (a.lse != nullptr && d0 == 0) a.lse[qrow] = (L > 0.f) ? (M * kLn2 + logf(L)) : -INFINITY;
}

// The CTA-level tail shared by both paths: merge the consumer warps' states
// (already in shared memory), then either write the output (one split) or the
// partial + ticket, with the last CTA of the unit merging all partials.
// `scratch` is free shared memory of at least 2 * kMaxGroup * n_splits + 16
// floats (the merge buffer may be reused once the warp merge is done).
template <typename T>
__device__ void decode_tail(const DecodeArgs& a, DecodeSmemTail& st, const float* obuf, float* scratch, int s, int h,
                            int split) {
  const int tid = threadIdx.x;
  const int64_t unit = static_cast<int64_t>(s) * a.hkv + h;
  // 8 heads x 16 eight-dim pieces = 128 items; threads 0..127
  const int head = tid >> 4;
  const int d0 = (tid & 15) * 8;
  const bool worker = tid < 128 && head < a.grp;
  float M = -INFINITY, L = 0.f, acc[8];
  if (worker) merge_states(kDecConsumers, &st.wm[0][0], &st.wl[0][0], kMaxGroup, obuf, kMaxGroup * kOStride, head,
                           d0, M, L, acc);
  if (a.n_splits == 1) {
    if (worker) write_final<T>(a, s, h, head, d0, M, L, acc);
    return;
  }
  float* part = a.partials + (unit * a.n_splits + split) * kPartFloats;
  if (worker) {
    if (d0 == 0) {
      part[head] = M;
      part[kMaxGroup + head] = L;
    }
    float* po = part + 2 * kMaxGroup + head * kHeadDim + d0;
    reinterpret_cast<float4*>(po)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    reinterpret_cast<float4*>(po)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.tickets[unit], 1);
    st.is_last = (prev == a.n_splits - 1);
  }
  __syncthreads();
  if (!st.is_last) return;
  __threadfence();
  // Last CTA of the unit. (1) every (split, head) max and sum, in parallel.
  const int n = a.n_splits;
  const float* base = a.partials + unit * n * kPartFloats;
  float* fm = scratch;                        // [n][8]: max, then the scale factor 2^(m_i - M)
  float* fl = scratch + n * kMaxGroup;        // [n][8]: sums
  float* tot = scratch + 2 * n * kMaxGroup;   // [8] M, [8] L
  for (int i = tid; i < n * kMaxGroup; i += blockDim.x) {
    const int sp = i / kMaxGroup, hh = i % kMaxGroup;
    fm[i] = __ldcg(base + sp * kPartFloats + hh);
    fl[i] = __ldcg(base + sp * kPartFloats + kMaxGroup + hh);
  }
  __syncthreads();
  // (2) per head: global max, factors and total sum
  if (tid < kMaxGroup) {
    float Mx = -INFINITY;
    for (int i = 0; i < n; ++i) Mx = fmaxf(Mx, fm[i * kMaxGroup + tid]);
    float Lx = 0.f;
    for (int i = 0; i < n; ++i) {
      const float f = (Mx == -INFINITY) ? 0.f : exp2f(fm[i * kMaxGroup + tid] - Mx);
      fm[i * kMaxGroup + tid] = f;
      Lx += f * fl[i * kMaxGroup + tid];
    }
    tot[tid] = Mx;
    tot[kMaxGroup + tid] = Lx;
  }
  __syncthreads();
  // (3) weighted sum of the partial outputs, several splits in flight
  if (worker) {
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = 0.f;
    const float* po = base + 2 * kMaxGroup + head * kHeadDim + d0;
    int i = 0;
    for (; i + 4 <= n; i += 4) {
      float4 u[4], v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        u[j] = __ldcg(reinterpret_cast<const float4*>(po + (i + j) * kPartFloats));
        v[j] = __ldcg(reinterpret_cast<const float4*>(po + (i + j) * kPartFloats + 4));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float f = fm[(i + j) * kMaxGroup + head];
        o[0] = fmaf(f, u[j].x, o[0]); o[1] = fmaf(f, u[j].y, o[1]); o[2] = fmaf(f, u[j].z, o[2]);
        o[3] = fmaf(f, u[j].w, o[3]); o[4] = fmaf(f, v[j].x, o[4]); o[5] = fmaf(f, v[j].y, o[5]);
        o[6] = fmaf(f, v[j].z, o[6]); o[7] = fmaf(f, v[j].w, o[7]);
      }
    }
    for (; i < n; ++i) {
      const float4 u = __ldcg(reinterpret_cast<const float4*>(po + i * kPartFloats));
      const float4 v = __ldcg(reinterpret_cast<const float4*>(po + i * kPartFloats + 4));
      const float f = fm[i * kMaxGroup + head];
      o[0] = fmaf(f, u.x, o[0]); o[1] = fmaf(f, u.y, o[1]); o[2] = fmaf(f, u.z, o[2]); o[3] = fmaf(f, u.w, o[3]);
      o[4] = fmaf(f, v.x, o[4]); o[5] = fmaf(f, v.y, o[5]); o[6] = fmaf(f, v.z, o[6]); o[7] = fmaf(f, v.w, o[7]);
    }
    write_final<T>(a, s, h, head, d0, tot[head], tot[kMaxGroup + head], o);
  }
  if (tid == 0) a.tickets[unit] = 0;  // ready for the next call
}

// Split-K combine inside a thread-block cluster (the unit's n_splits CTAs, n a
// power of two <= 16): each CTA merges its warps into `xch` (M[8], L[8],
// O[8][128]); after a cluster barrier, CTA r produces the output pieces
// r, r + n, ... (a piece = 8 dims of one head) by reading every CTA's `xch`
// through distributed shared memory, one source per lane of an n-lane group,
// reduced with shuffles. A second barrier keeps each `xch` alive until read.
template <typename T>
__device__ void decode_tail_cluster(const DecodeArgs& a, DecodeSmemTail& st, const float* obuf, float* xch, int s,
                                    int h) {
  const int tid = threadIdx.x;
  {
    const int head = tid >> 4;
    const int d0 = (tid & 15) * 8;
    if (tid < 128 && head < a.grp) {
      float M, L, acc[8];
      merge_states(kDecConsumers, &st.wm[0][0], &st.wl[0][0], kMaxGroup, obuf, kMaxGroup * kOStride, head, d0, M, L,
                   acc);
      if (d0 == 0) {
        xch[head] = M;
        xch[kMaxGroup + head] = L;
      }
      float* dst = xch + 2 * kMaxGroup + head * kHeadDim + d0;
      reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
  cluster_sync();
  if (tid < 128) {
    const int n = a.n_splits;
    const uint32_t r = cluster_ctarank();
    const int pieces = a.grp * 16;
    const int j = tid / n, i = tid % n;
    const int piece = j * n + static_cast<int>(r);
    const bool live = piece < pieces;
    const int head = live ? piece >> 4 : 0;
    const int d0 = live ? (piece & 15) * 8 : 0;
    float Mi = -INFINITY, Li = 0.f;
    float4 oa = make_float4(0.f, 0.f, 0.f, 0.f), ob = oa;
    if (live) {
      const uint32_t base = dsmem_addr(smem_u32(xch), static_cast<uint32_t>(i));
      Mi = ld_dsmem(base + 4u * head);
      Li = ld_dsmem(base + 4u * (kMaxGroup + head));
      oa = ld_dsmem4(base + 4u * (2 * kMaxGroup + head * kHeadDim + d0));
      ob = ld_dsmem4(base + 4u * (2 * kMaxGroup + head * kHeadDim + d0 + 4));
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
      const float o[8] = {v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8]};
      write_final<T>(a, s, h, head, d0, Mx, v[0], o);
    }
  }
  cluster_sync();
}

// Collects this CTA's list of valid blocks into shared memory (warp 0: one
// entry per lane, compacted with a ballot).
__device__ inline void gather_block_list(const DecodeArgs& a, const KvView& kv, DecodeSmemTail& st, int s, int h,
                                         int split, int64_t nb) {
  const int tid = threadIdx.x;
  if (tid >= 32) return;
  const int lane = tid;
  int n = 0;
  if (a.idx != nullptr) {
    const int32_t* list = a.idx + (static_cast<int64_t>(s) * a.hkv + h) * a.k_total;
    const int lo = split * a.bps;
    const int hi = min(a.k_total, lo + a.bps);
    for (int base = lo; base < hi; base += 32) {
      const int i = base + lane;
      const int32_t b = i < hi ? list[i] : -1;
      if (b >= nb) set_status(a.status, MSA_ERR_DEVICE_BOUNDS, kIdDecode);
      const bool ok = b >= 0 && b < nb;
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) st.blocks[n + __popc(m & ((1u << lane) - 1u))] = b;
      n += __popc(m);
    }
  } else {
    const int64_t lo = static_cast<int64_t>(split) * a.bps;
    const int64_t hi = min(nb, lo + a.bps);
    n = hi > lo ? static_cast<int>(hi - lo) : 0;
    if (lane == 0) st.dense_lo = static_cast<int32_t>(lo);
  }
  if (lane == 0) st.n_blocks = n;
}

// ---------------------------------------------------------------------------
// bf16 kernel. grid (n_splits, Hkv, batch), kDecThreads threads.
// ---------------------------------------------------------------------------
template <int kStages>
__global__ void __launch_bounds__(kDecThreads) decode_bf16_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                 const __grid_constant__ CUtensorMap tmv, KvView kv,
                                                                 DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_align1024(smem_raw);
  DecodeSmemTail& st = *reinterpret_cast<DecodeSmemTail*>(ring + kStages * kStageBytes);

  const int split = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&st.full[i], 1);
      mbar_init(&st.empty[i], kDecConsumers);
    }
    fence_mbar_init();
  }
  if (warp == kDecConsumers && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  pdl_wait();  // the index lists (and every other input) come from earlier work
  const int64_t len = kv.seq_len(s, a.status, kIdDecode);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  gather_block_list(a, kv, st, s, h, split, nb);
  __syncthreads();
  const int nblk = st.n_blocks;

  const int g = lane >> 2, c = lane & 3;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  if (warp == kDecConsumers) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        const int stg = i % kStages;
        if (i >= kStages && !mbar_wait(&st.empty[stg], ((i / kStages) - 1) & 1, a.status, kIdDecode)) break;
        issued = i + 1;
        const int64_t row = kv.block_row(s, h, a.idx ? st.blocks[i] : st.dense_lo + i, a.status, kIdDecode);
        uint8_t* dst = ring + stg * kStageBytes;
        mbar_arrive_expect_tx(&st.full[stg], kStageBytes);
        const int32_t y = static_cast<int32_t>(row < 0 ? 0 : row);
        tma_load_2d(dst, &tmk, 0, y, &st.full[stg]);
        tma_load_2d(dst + 8192, &tmk, 64, y, &st.full[stg]);
        tma_load_2d(dst + 16384, &tmv, 0, y, &st.full[stg]);
        tma_load_2d(dst + 24576, &tmv, 64, y, &st.full[stg]);
      }
      mbar_drain(st.full, kStages, issued, a.status, kIdDecode);
    }
  } else {
    // ---------------- consumers ----------------
    // Q^T fragments (B operand of S = K Q^T): head g, dims 16kk + 2c (+1), +8 (+9)
    uint32_t qb[8][2];
    {
      const bool live = g < a.grp;
      const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                  (static_cast<int64_t>(s) * a.hq + h * a.grp + (live ? g : 0)) * kHeadDim;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * c) : 0u;
        qb[kk][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * c + 8) : 0u;
      }
    }
    const int krow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;  // K ldmatrix row
    const int kchunk = lane >> 4;
    const int vrow = 16 * warp + (lane & 7) + ((lane >> 4) & 1) * 8;  // V ldmatrix.trans row
    const int vchunk = (lane >> 3) & 1;
    for (int i = 0; i < nblk; ++i) {
      const int stg = i % kStages;
      if (!mbar_wait_warp(&st.full[stg], (i / kStages) & 1, a.status, kIdDecode)) break;
      const uint32_t kbase = smem_u32(ring + stg * kStageBytes);
      const uint32_t vbase = kbase + 16384;
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + (kk >> 2) * 8192 + swz128(krow, (kk & 3) * 2 + kchunk), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      const int64_t tok = static_cast<int64_t>(a.idx ? st.blocks[i] : st.dense_lo + i) * kBlock + 16 * warp + g;
      const bool v0 = tok < len, v1 = tok + 8 < len;
      const float s0 = v0 ? sacc[0] * a.scale_log2 : -INFINITY;  // token g,   head 2c
      const float s1 = v0 ? sacc[1] * a.scale_log2 : -INFINITY;  // token g,   head 2c+1
      const float s2 = v1 ? sacc[2] * a.scale_log2 : -INFINITY;  // token g+8, head 2c
      const float s3 = v1 ? sacc[3] * a.scale_log2 : -INFINITY;  // token g+8, head 2c+1
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float r0 = mn0 == -INFINITY ? 0.f : mn0;
      const float r1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - r0), al1 = exp2f(m1 - r1);
      const float p0 = exp2f(s0 - r0), p2 = exp2f(s2 - r0);
      const float p1 = exp2f(s1 - r1), p3 = exp2f(s3 - r1);
      l0 = l0 * al0 + p0 + p2;
      l1 = l1 * al1 + p1 + p3;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o[j][0] *= al0; o[j][1] *= al1; o[j][2] *= al0; o[j][3] *= al1;
      }
      const uint32_t pb0 = movm_t(pack_bf16(p0, p1));  // tokens 0-7  -> (k = 2c.., n = head g)
      const uint32_t pb1 = movm_t(pack_bf16(p2, p3));  // tokens 8-15
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + (j >> 2) * 8192 + swz128(vrow, (j & 3) * 2 + vchunk), a0, a1, a2, a3);
        mma_bf16(o[j], a0, a1, a2, a3, pb0, pb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&st.empty[stg]);
    }
    // l partial sums live on the 8 lanes that share c
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
  pdl_trigger();    // the next kernel may start its set-up
  __syncthreads();  // every consumer is done with the ring: reuse it for the merge
  if (warp < kDecConsumers) {
    float* obuf = reinterpret_cast<float*>(ring) + warp * kMaxGroup * kOStride;
    if (g == 0) {
      st.wm[warp][2 * c] = m0;
      st.wm[warp][2 * c + 1] = m1;
      st.wl[warp][2 * c] = l0;
      st.wl[warp][2 * c + 1] = l1;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      obuf[(2 * c) * kOStride + 16 * j + g] = o[j][0];
      obuf[(2 * c + 1) * kOStride + 16 * j + g] = o[j][1];
      obuf[(2 * c) * kOStride + 16 * j + g + 8] = o[j][2];
      obuf[(2 * c + 1) * kOStride + 16 * j + g + 8] = o[j][3];
    }
  }
  __syncthreads();
  if (a.n_splits > 1) {
    decode_tail_cluster<__nv_bfloat16>(a, st, reinterpret_cast<const float*>(ring),
                                       reinterpret_cast<float*>(ring) + kDecConsumers * kMaxGroup * kOStride, s, h);
  } else {
    decode_tail<__nv_bfloat16>(a, st, reinterpret_cast<const float*>(ring),
                               reinterpret_cast<float*>(ring) + kDecConsumers * kMaxGroup * kOStride, s, h, split);
  }
}

// ---------------------------------------------------------------------------
// fp32 kernel (CUDA cores). grid (n_splits, Hkv, batch), kDecThreads threads;
// warps 0-3 compute, warp 4 idles until the merge.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kDecThreads) decode_f32_kernel(const float* __restrict__ k,
                                                                const float* __restrict__ v, KvView kv,
                                                                DecodeArgs a) {
  __shared__ __align__(16) float obuf[kDecConsumers * kMaxGroup * kOStride];
  __shared__ __align__(16) float merge_scratch[2 * kMaxGroup * kMaxSplits + 2 * kMaxGroup];
  __shared__ DecodeSmemTail st;
  const int split = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t len = kv.seq_len(s, a.status, kIdDecode);
  const int64_t nb = (len + kBlock - 1) / kBlock;
  gather_block_list(a, kv, st, s, h, split, nb);
  __syncthreads();
  const int nblk = st.n_blocks;
  if (warp < kDecConsumers) {
    const int grp = a.grp;
    const float* qbase = reinterpret_cast<const float*>(a.q) + (static_cast<int64_t>(s) * a.hq + h * grp) * kHeadDim;
    float qv[kMaxGroup][4], ov[kMaxGroup][4], m[kMaxGroup], l[kMaxGroup];
#pragma unroll
    for (int j = 0; j < kMaxGroup; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qv[j][i] = j < grp ? qbase[j * kHeadDim + 4 * lane + i] : 0.f;
        ov[j][i] = 0.f;
      }
    }
    for (int bi = 0; bi < nblk; ++bi) {
      const int32_t blk = a.idx ? st.blocks[bi] : st.dense_lo + bi;
      const int64_t row0 = kv.block_row(s, h, blk, a.status, kIdDecode);
      if (row0 < 0) continue;
      for (int t = 16 * warp; t < 16 * warp + 16; ++t) {
        const int64_t tok = static_cast<int64_t>(blk) * kBlock + t;
        if (tok >= len) break;
        const float4 kk = *reinterpret_cast<const float4*>(k + (row0 + t) * kHeadDim + 4 * lane);
        const float4 vv = *reinterpret_cast<const float4*>(v + (row0 + t) * kHeadDim + 4 * lane);
#pragma unroll
        for (int j = 0; j < kMaxGroup; ++j) {
          if (j >= grp) break;
          float part = qv[j][0] * kk.x + qv[j][1] * kk.y + qv[j][2] * kk.z + qv[j][3] * kk.w;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
          const float z = part * a.scale_log2;
          const float mn = fmaxf(m[j], z);
          const float al = exp2f(m[j] - mn);
          const float p = exp2f(z - mn);
          l[j] = l[j] * al + p;
          m[j] = mn;
          ov[j][0] = ov[j][0] * al + p * vv.x;
          ov[j][1] = ov[j][1] * al + p * vv.y;
          ov[j][2] = ov[j][2] * al + p * vv.z;
          ov[j][3] = ov[j][3] * al + p * vv.w;
        }
      }
    }
    float* ob = obuf + warp * kMaxGroup * kOStride;
#pragma unroll
    for (int j = 0; j < kMaxGroup; ++j) {
      if (lane == 0) {
        st.wm[warp][j] = m[j];
        st.wl[warp][j] = l[j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) ob[j * kOStride + 4 * lane + i] = ov[j][i];
    }
  }
  __syncthreads();
  decode_tail<float>(a, st, obuf, merge_scratch, s, h, split);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
constexpr int kDecStages = 3;

size_t decode_smem_bytes() { return 1024 + kDecStages * kStageBytes + sizeof(DecodeSmemTail); }

cudaError_t set_decode_smem() {
  cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel<kDecStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(decode_smem_bytes()));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_bf16_kernel<kDecStages>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_bf16_kernel<kDecStages>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_f32_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// Split heuristic: fill the resident CTA slots (two 3-stage CTAs per SM) in a
// single wave: units x splits <= 2 x SMs where possible, at most
// kMaxListPerCta list entries per CTA. The bf16 kernel combines its splits in
// a thread-block cluster, so there the split count is a power of two <= 16;
// the fp32 kernel combines through global memory (up to kMaxSplits).
void decode_splits(int64_t units, int64_t list_len, int num_sms, bool cluster, bool dense, int* n_splits, int* bps) {
  const int64_t slots = 2LL * num_sms;
  int64_t want = units >= slots ? 1 : slots / units;
  if (want < 1) want = 1;
  if (cluster) {
    int64_t p = 1;
    while (p * 2 <= want && p * 2 <= 16) p *= 2;
    while (p < 16 && (list_len + p - 1) / p > kMaxListPerCta) p *= 2;
    *n_splits = static_cast<int>(p);
    *bps = static_cast<int>((list_len + p - 1) / p);
    if (*bps < 1) *bps = 1;
    return;
  }
  int64_t b = (list_len + want - 1) / want;
  if (b < 1) b = 1;
  if (!dense && b > kMaxListPerCta) b = kMaxListPerCta;
  int64_t ns = (list_len + b - 1) / b;
  if (ns > kMaxSplits) {
    b = (list_len + kMaxSplits - 1) / kMaxSplits;
    ns = (list_len + b - 1) / b;
  }
  *bps = static_cast<int>(b);
  *n_splits = static_cast<int>(ns < 1 ? 1 : ns);
}

size_t decode_partials_bytes(int64_t units, int n_splits) {
  return static_cast<size_t>(units) * n_splits * kPartFloats * sizeof(float);
}

cudaError_t launch_decode_bf16(const CUtensorMap& tmk, const CUtensorMap& tmv, const KvView& kv, int batch,
                               const DecodeArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, kv.hkv, batch);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = decode_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.n_splits;  // the unit's splits form one cluster
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_bf16_kernel<kDecStages>, tmk, tmv, kv, a);
}

cudaError_t launch_decode_f32(const float* k, const float* v, const KvView& kv, int batch, const DecodeArgs& a,
                              cudaStream_t stream) {
  dim3 grid(a.n_splits, kv.hkv, batch);
  decode_f32_kernel<<<grid, kDecThreads, 0, stream>>>(k, v, kv, a);
  return cudaGetLastError();
}

}  // namespace msa
