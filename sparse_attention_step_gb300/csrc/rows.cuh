// Reading 8-dimension slices of summary-key rows and query heads (bf16 or
// fp32) and dotting them with an fp32 index query slice.
#pragma once

#include "common.cuh"

namespace msa {

// One summary row slice (8 dims) kept in its storage form until used.
template <typename T>
struct RawRow;
template <>
struct RawRow<__nv_bfloat16> {
  uint4 w;
  __device__ void load(const __nv_bfloat16* p) { w = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ float dot(const float (&qi)[8]) const {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(qi[2 * i], __uint_as_float(v[i] << 16), acc);
      acc = fmaf(qi[2 * i + 1], __uint_as_float(v[i] & 0xFFFF0000u), acc);
    }
    return acc;
  }
  __device__ void add_to(float (&acc)[8]) const {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += __uint_as_float(v[i] << 16);
      acc[2 * i + 1] += __uint_as_float(v[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct RawRow<float> {
  float4 a, b;
  __device__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ float dot(const float (&qi)[8]) const {
    float acc = 0.f;
    acc = fmaf(qi[0], a.x, acc); acc = fmaf(qi[1], a.y, acc); acc = fmaf(qi[2], a.z, acc); acc = fmaf(qi[3], a.w, acc);
    acc = fmaf(qi[4], b.x, acc); acc = fmaf(qi[5], b.y, acc); acc = fmaf(qi[6], b.z, acc); acc = fmaf(qi[7], b.w, acc);
    return acc;
  }
  __device__ void add_to(float (&acc)[8]) const {
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
};

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

template <typename T>
struct SelRow;  // 8 dims of a staged summary row, dotted with q_idx
template <>
struct SelRow<__nv_bfloat16> {
  static constexpr int kBytes = kHeadDim * 2;
  __device__ static float dot(const uint8_t* row, int e, const float (&qi)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * e);
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(qi[2 * i], __uint_as_float(v[i] << 16), acc);
      acc = fmaf(qi[2 * i + 1], __uint_as_float(v[i] & 0xFFFF0000u), acc);
    }
    return acc;
  }
};
template <>
struct SelRow<float> {
  static constexpr int kBytes = kHeadDim * 4;
  __device__ static float dot(const uint8_t* row, int e, const float (&qi)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(row + 32 * e);
    const float4 b = *reinterpret_cast<const float4*>(row + 32 * e + 16);
    float acc = 0.f;
    acc = fmaf(qi[0], a.x, acc); acc = fmaf(qi[1], a.y, acc); acc = fmaf(qi[2], a.z, acc); acc = fmaf(qi[3], a.w, acc);
    acc = fmaf(qi[4], b.x, acc); acc = fmaf(qi[5], b.y, acc); acc = fmaf(qi[6], b.z, acc); acc = fmaf(qi[7], b.w, acc);
    return acc;
  }
};

}  // namespace msa
