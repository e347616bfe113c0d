// Small device helpers shared by the attention kernels.
#pragma once
#include <cmath>

namespace ditattn {

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Max of 32 values with eight independent accumulators.
__device__ __forceinline__ float rowmax32(const float* s) {
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = fmaxf(s[2 * j], s[2 * j + 1]);
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = max3f(a[j], s[16 + 2 * j], s[16 + 2 * j + 1]);
  return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// Max of 64 values with eight independent accumulators.
__device__ __forceinline__ float rowmax64(const float* s) {
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = fmaxf(s[2 * j], s[2 * j + 1]);
#pragma unroll
  for (int k = 16; k < 64; k += 16)
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = max3f(a[j], s[k + 2 * j], s[k + 2 * j + 1]);
  return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// Max of 128 values with eight independent accumulators.
__device__ __forceinline__ float rowmax128(const float* s) {
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = fmaxf(s[2 * j], s[2 * j + 1]);
#pragma unroll
  for (int k = 16; k < 128; k += 16)
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = max3f(a[j], s[k + 2 * j], s[k + 2 * j + 1]);
  return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// Max of one K-scale group of G consecutive columns.
template <int G>
__device__ __forceinline__ float groupmax(const float* s) {
  if constexpr (G == 4) {
    return fmaxf(max3f(s[0], s[1], s[2]), s[3]);
  } else {
    static_assert(G == 16, "group sizes 4 and 16");
    const float a = max3f(s[0], s[1], s[2]), b = max3f(s[3], s[4], s[5]), c = max3f(s[6], s[7], s[8]);
    const float d = max3f(s[9], s[10], s[11]), e = max3f(s[12], s[13], s[14]);
    return max3f(max3f(a, b, c), max3f(d, e, s[15]), -INFINITY);
  }
}

}  // namespace ditattn
