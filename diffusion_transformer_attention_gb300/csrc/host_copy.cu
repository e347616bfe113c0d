// Row copies between page-locked host memory and device memory, driven by the SMs.
//
// dit_attn_fwd_host moves head slices of [B, S, H, 128] tensors: rows of a few heads' 256-byte
// slices at a pitch of H x 256 bytes. The copy engines move such 2-D slices at well below the host
// link's rate when the rows are narrow (measured on GB300: 70 GB/s for 256-byte rows, 168 GB/s for
// 1,280-byte rows, against 211 GB/s for a 1-D copy), while SM loads and stores through the device
// mapping of page-locked host memory reach the link's rate for any row width. The entry point uses
// this kernel only for the transfers that no attention kernel hides (its first group's inputs and its
// last group's output), when no attention kernel is running.
#include <cuda_runtime.h>

#include <cstdint>

#include "ditattn_internal.h"

namespace ditattn {
namespace {

// `rows` rows of `vec` 16-byte vectors from src (row pitch src_pitch vectors) to dst (row pitch
// dst_pitch vectors).
__global__ void __launch_bounds__(256) copy_rows_kernel(const uint4* __restrict__ src, long long src_pitch,
                                                        uint4* __restrict__ dst, long long dst_pitch, int vec,
                                                        long long rows) {
  const long long n = rows * vec;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const long long r = i / vec, c = i - r * vec;
    dst[r * dst_pitch + c] = src[r * src_pitch + c];
  }
}

}  // namespace

cudaError_t launch_copy_rows(const void* src, size_t src_pitch, void* dst, size_t dst_pitch, size_t width,
                             size_t rows, cudaStream_t stream) {
  if (rows == 0 || width == 0) return cudaSuccess;
  if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | src_pitch | dst_pitch | width) & 15u) !=
          0 ||
      width > src_pitch || width > dst_pitch)
    return cudaErrorInvalidValue;
  const long long vec = (long long)(width / 16), n = vec * (long long)rows;
  long long grid = (n + 255) / 256;
  if (grid > 152LL * 8) grid = 152LL * 8;  // a few CTAs per SM; the loop covers the rest
  copy_rows_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint4*>(src), (long long)(src_pitch / 16),
                                                       static_cast<uint4*>(dst), (long long)(dst_pitch / 16),
                                                       (int)vec, (long long)rows);
  return cudaGetLastError();
}

}  // namespace ditattn
