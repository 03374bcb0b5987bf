// Step 1a: block summary keys ("MiniMax goes sparse", §1 Step 1, block pooling
// in the index branch). The summary of a complete 64-token block is the mean of
// its keys, summed in fp32 in row order and scaled once by 1/64, then rounded
// to nearest even into the KV dtype.
//
// Bandwidth-bound: every key byte is read once, 1/64 of it is written. A
// half-warp owns one block: lane e holds dims [8e, 8e+8) (16 B of bf16) and
// walks the 64 rows in order, so every row read by the half-warp is one
// contiguous 256-byte segment.
#include "kernels.cuh"

namespace msa {

constexpr int kPoolThreads = 256;
constexpr int kPoolBlocksPerCta = kPoolThreads / 16;

template <typename T>
struct Vec8;  // eight consecutive head-dim elements of one row

template <>
struct Vec8<__nv_bfloat16> {
  uint4 raw;
  __device__ void load(const __nv_bfloat16* p) { raw = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ void add_to(float (&acc)[8]) const {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += __uint_as_float(w[i] << 16);
      acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&x)[8]) {
    uint4 o;
    o.x = pack_bf16(x[0], x[1]);
    o.y = pack_bf16(x[2], x[3]);
    o.z = pack_bf16(x[4], x[5]);
    o.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4*>(p) = o;
  }
};

template <>
struct Vec8<float> {
  float4 a, b;
  __device__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ void add_to(float (&acc)[8]) const {
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  __device__ static void store(float* p, const float (&x)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

// grid: (ceil(block range / 16), Hkv, batch). newest_only: grid (1, Hkv,
// batch) and each sequence pools only its newest block, when that block has
// just filled (seq_len a multiple of 64).
template <typename T>
__global__ void __launch_bounds__(kPoolThreads) pool_block_keys_kernel(const T* __restrict__ k, KvView kv,
                                                                      int64_t first_block, int64_t n_blocks,
                                                                      int newest_only, T* __restrict__ pooled,
                                                                      int32_t* status) {
  const int s = blockIdx.z;
  const int h = blockIdx.y;
  const int e = threadIdx.x & 15;
  const int64_t len = kv.seq_len(s, status, kIdPool);
  int64_t b = first_block + static_cast<int64_t>(blockIdx.x) * kPoolBlocksPerCta + (threadIdx.x >> 4);
  if (newest_only) {
    if (threadIdx.x >= 16 || len == 0 || len % kBlock != 0) return;
    b = len / kBlock - 1;
  } else if (n_blocks >= 0 && b >= first_block + n_blocks) {
    return;
  }
  if ((b + 1) * kBlock > len) return;  // partial or absent block: not pooled
  const int64_t row = kv.block_row(s, h, b, status, kIdPool);
  const int64_t prow = kv.pooled_row(s, h, b);
  if (row < 0) return;  // bad page: reported, its summary not written
  const T* src = k + row * kHeadDim + 8 * e;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 1
  for (int t0 = 0; t0 < kBlock; t0 += 16) {
    Vec8<T> v[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t].load(src + (t0 + t) * kHeadDim);
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t].add_to(acc);  // row order
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] *= (1.0f / kBlock);
  Vec8<T>::store(pooled + prow * kHeadDim + 8 * e, acc);
}

template <typename T>
cudaError_t launch_pool(const T* k, const KvView& kv, int batch, int64_t first_block, int64_t n_blocks,
                        T* pooled, int32_t* status, cudaStream_t stream) {
  int64_t span = kv.max_blocks();
  span -= first_block;
  if (n_blocks >= 0 && n_blocks < span) span = n_blocks;
  if (span <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((span + kPoolBlocksPerCta - 1) / kPoolBlocksPerCta), kv.hkv, batch);
  pool_block_keys_kernel<T><<<grid, kPoolThreads, 0, stream>>>(k, kv, first_block, n_blocks, 0, pooled, status);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pool_newest(const T* k, const KvView& kv, int batch, T* pooled, int32_t* status,
                               cudaStream_t stream) {
  pool_block_keys_kernel<T><<<dim3(1, kv.hkv, batch), kPoolThreads, 0, stream>>>(k, kv, 0, -1, 1, pooled, status);
  return cudaGetLastError();
}

template cudaError_t launch_pool<__nv_bfloat16>(const __nv_bfloat16*, const KvView&, int, int64_t, int64_t,
                                                __nv_bfloat16*, int32_t*, cudaStream_t);
template cudaError_t launch_pool<float>(const float*, const KvView&, int, int64_t, int64_t, float*, int32_t*,
                                        cudaStream_t);
template cudaError_t launch_pool_newest<__nv_bfloat16>(const __nv_bfloat16*, const KvView&, int, __nv_bfloat16*,
                                                       int32_t*, cudaStream_t);
template cudaError_t launch_pool_newest<float>(const float*, const KvView&, int, float*, int32_t*, cudaStream_t);

}  // namespace msa
