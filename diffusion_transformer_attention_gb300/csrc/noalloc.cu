// sage_quantize_qkv_noalloc: the SAGE quantize prepass with its scratch memory held by the
// library itself, for callers that cannot allocate device memory when they call us.
//
// The regular sage_quantize_qkv needs a caller-provided workspace for the per-chunk partial
// sums of K and partial maxima of |V|. Some callers cannot provide one: a plugin whose host
// framework owns the whole device memory pool and hands it no allocator, or code running in a
// latency-critical loop where cudaMalloc (which may synchronize the whole device) is not
// allowed. This entry point takes the same inputs and outputs but keeps the partials in a
// fixed-size array that every GPU loading this library reserves once, until process exit.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/ditattn.h"
#include "ditattn_internal.h"

using namespace ditattn;

namespace {

// Largest scratch this entry point can use: the partial sums (8 bytes) and maxima (4 bytes) of
// B * Hkv * ceil(Skv / 1024) chunks of 128 channels, each part rounded up to 256 bytes.
constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) uint8_t g_prepass_scratch[kScratchBytes];

// Device address of g_prepass_scratch, looked up once per device. In host code the array's
// name only stands in for the symbol; it is not a device address. Only a successful lookup is
// cached: a failure (for example, no room to load the module that holds the array) is reported
// and tried again on the next call.
uint8_t* g_addr[64];
std::mutex g_addr_mu;

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

dit_status scratch_for_current_device(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return DIT_E_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (g_addr[dev] == nullptr) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return DIT_E_CUDA;
    }
    if (!(prop.major == 10 && prop.minor == 3)) return DIT_E_UNSUPPORTED;
    // With lazy module loading this is the call that loads the module and so reserves the array.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prepass_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return DIT_E_CUDA;
    }
    g_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_addr[dev];
  return DIT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

dit_status sage_quantize_qkv_noalloc(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Sq,
                                     int Skv, int qk_dtype, int q_block, int k_block, void* q_codes, void* k_codes,
                                     void* v_codes, float* q_scale, float* k_scale, float* v_scale, float* k_mean,
                                     void* stream) {
  // The same argument checks as sage_quantize_qkv, in an order that launches nothing for a problem
  // too large for the fixed scratch whatever its pointers are.
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || (qk_dtype != DIT_QK_INT8 && qk_dtype != DIT_QK_FP8_E4M3) ||
      !valid_mode(DIT_MODE_SAGE, qk_dtype, q_block, k_block, 0.0f))
    return DIT_E_INVALID_ARG;
  if (B == 0) return DIT_OK;
  const size_t n = (size_t)B * Hkv * stats_chunks(Skv) * kHeadDim;
  const size_t sum_bytes = round256(n * 8);
  if (sum_bytes + round256(n * 4) > kScratchBytes) return DIT_E_WORKSPACE;  // beyond the fixed scratch
  const void* ptrs[] = {k, v, k_codes, v_codes, k_scale, v_scale, k_mean};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return DIT_E_INVALID_ARG;
  if (Sq > 0 && (!q || !q_codes || !q_scale || !aligned16(q) || !aligned16(q_codes))) return DIT_E_INVALID_ARG;
  uint8_t* scratch = nullptr;
  const dit_status ds = scratch_for_current_device(&scratch);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The partial kernel writes every sum and maximum the final kernel reads, so the scratch
  // needs no clearing between calls.
  const int code_out = (qk_dtype == DIT_QK_INT8) ? CODE_I8 : CODE_E4M3;
  cudaError_t e = launch_kv_stats(k, v, B, Hkv, Skv, reinterpret_cast<double*>(scratch),
                                  reinterpret_cast<float*>(scratch + sum_bytes), k_mean, v_scale, st);
  if (e == cudaSuccess && Sq > 0) e = launch_quant_q(q, B, Hq, Sq, q_block, code_out, q_codes, q_scale, st, true);
  if (e == cudaSuccess)
    e = launch_quant_kv(k, v, B, Hkv, Skv, k_block, code_out, k_mean, v_scale, k_codes, k_scale, v_codes, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DIT_E_CUDA;
  }
  return DIT_OK;
}

}  // extern "C"
