// C-ABI entry points (include/ditattn.h): argument validation, workspace layout, TMA tensor-map
// encoding and the launch sequence. Arguments are validated on the host before any CUDA call,
// so a rejected call has no side effects and needs no GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/ditattn.h"
#include "ditattn_internal.h"

using namespace ditattn;

namespace {

constexpr int kAbiVersion = 4;
constexpr unsigned long long kWaitBudgetNs = 4000000000ull;  // far beyond any legitimate wait

__device__ int g_device_error = 0;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

struct SageLayout {
  size_t q_codes, k_codes, v_codes, q_scale, k_scale, v_scale, k_mean, psum, pmax, gs, total;
};

// Workspace of the all-in-one call. QK16PV8 (BF16 Q/K) needs only the V codes, V scales and the
// V-absmax partials; its Q/K regions have size zero. MXFP8 holds 1-byte Q/K codes and, in the
// scale regions, 4 E8M0 bytes per token and head; NVFP4 holds half-byte codes, 8 E4M3 bytes per
// token and head and the two tensor scales. Neither has a K mean.
SageLayout sage_layout(int B, int Hq, int Hkv, int Sq, int Skv, int qk_dtype, int q_block, int k_block) {
  SageLayout L{};
  const bool qk16 = (qk_dtype == DIT_QK_BF16);
  const bool mx = (qk_dtype == DIT_QK_MXFP8);
  const bool nv = (qk_dtype == DIT_QK_NVFP4);
  // bytes per 128-channel row of codes: INT8 codes are held as exact fp16, NVFP4 packs two per byte
  const size_t row_bytes = qk16 ? 0 : (qk_dtype == DIT_QK_INT8) ? 256 : nv ? 64 : 128;
  const size_t sf_row = mx ? 4 : 8;  // block-scale bytes per token and head
  const size_t q_scale_bytes =
      qk16 ? 0 : (mx || nv) ? (size_t)B * Hq * Sq * sf_row : (size_t)B * Hq * ceil_div(Sq, q_block) * 4;
  const size_t k_scale_bytes =
      qk16 ? 0 : (mx || nv) ? (size_t)B * Hkv * Skv * sf_row : (size_t)B * Hkv * ceil_div(Skv, k_block) * 4;
  const bool smooth = !qk16 && !mx && !nv;
  size_t off = 0;
  L.q_codes = off; off = align256(off + (size_t)B * Sq * Hq * row_bytes);
  L.k_codes = off; off = align256(off + (size_t)B * Skv * Hkv * row_bytes);
  L.v_codes = off; off = align256(off + (size_t)B * Skv * Hkv * kHeadDim);
  L.q_scale = off; off = align256(off + q_scale_bytes);
  L.k_scale = off; off = align256(off + k_scale_bytes);
  L.v_scale = off; off = align256(off + (size_t)B * Hkv * kHeadDim * 4);
  L.k_mean = off;  off = align256(off + (smooth ? (size_t)B * Hkv * kHeadDim * 4 : 0));
  L.psum = off;    off = align256(off + (smooth ? (size_t)B * Hkv * stats_chunks(Skv) * kHeadDim * 8 : 0));
  L.pmax = off;    off = align256(off + (size_t)B * Hkv * stats_chunks(Skv) * kHeadDim * 4);
  L.gs = off;      off = align256(off + (nv ? 2 * sizeof(float) : 0));
  L.total = off;
  return L;
}

size_t stats_bytes(int B, int Hkv, int Skv) {
  const size_t n = (size_t)B * Hkv * stats_chunks(Skv) * kHeadDim;
  return align256(n * 8) + align256(n * 4);
}

// ------------------------------------------------------------------ device checks and state
struct DeviceState {
  bool checked = false;
  bool supported = false;
  int* err = nullptr;
};
DeviceState g_dev[64];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

dit_status prepare_device(int** err_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return DIT_E_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.checked) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return DIT_E_UNSUPPORTED;
    }
    st.checked = true;
    st.supported = (prop.major == 10 && prop.minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
        cudaGetLastError();
        st.supported = false;
      }
      st.err = static_cast<int*>(p);
    }
    if (st.supported && g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        st.supported = false;
      } else {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
  }
  if (!st.supported) return DIT_E_UNSUPPORTED;
  *err_out = st.err;
  return DIT_OK;
}

// [B, S, H, 128] tensor as a 4-D map {128, S, H, B} with boxes of {box_inner, 128, 1, 1}
// (box_inner * element size = 128 bytes) and 128-byte swizzling. Hstride >= H is the head count of
// the tensor's rows: H heads starting at ptr form a slice of a [B, S, Hstride, 128] tensor.
// packed4: NVFP4 codes, two per byte: 64-byte rows as a {64, S, H, B} byte tensor, boxes of
// {64, 128, 1, 1} with 64-byte swizzling.
bool encode_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esize, int B, int S, int H,
                int Hstride, bool packed4 = false) {
  const cuuint64_t inner = packed4 ? kHeadDim / 2 : kHeadDim;
  const cuuint64_t dims[4] = {inner, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t row = inner * esize;
  const cuuint64_t strides[3] = {row * (cuuint64_t)Hstride, row, row * (cuuint64_t)Hstride * (cuuint64_t)S};
  const cuuint32_t box[4] = {(cuuint32_t)(packed4 ? 64 : 128 / esize), 128, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              packed4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Events and a second compute stream for dit_attn_fwd_host, created once per device on first use
// (the calls themselves create nothing): one event per chunk for "inputs copied" and "attention
// done", plus start and finish. Consecutive chunks' kernels alternate between the caller's compute
// stream and `aux`, so each kernel's last partial wave of CTAs overlaps the next one's first.
constexpr int kMaxHostChunks = 64;
struct HostEvents {
  bool ok = false;
  cudaStream_t aux;
  cudaEvent_t start, done, aux_done, h2d_done, in[kMaxHostChunks], comp[kMaxHostChunks];
};
HostEvents g_host_events[64];
std::mutex g_host_mu;
// Held by dit_attn_fwd_host while it queues a call's work: concurrent calls from several host threads
// then queue one after the other. Reusing the events is safe once a call is queued, since each stream
// wait binds to the record that precedes it at the time it is queued.
std::mutex g_host_call_mu;

HostEvents* host_events() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostEvents& h = g_host_events[dev];
  if (h.ok) return &h;
  // Only a complete set is kept; a failed attempt releases what it created and is retried on the
  // next call (a transient failure, e.g. out of memory, is not cached).
  HostEvents n;
  std::vector<cudaEvent_t> made;
  bool aux_made = cudaStreamCreateWithFlags(&n.aux, cudaStreamNonBlocking) == cudaSuccess;
  bool ok = aux_made;
  auto make = [&](cudaEvent_t* e) {
    if (ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess) {
      made.push_back(*e);
    } else {
      ok = false;
    }
  };
  make(&n.start);
  make(&n.done);
  make(&n.aux_done);
  make(&n.h2d_done);
  for (int i = 0; i < kMaxHostChunks; ++i) {
    make(&n.in[i]);
    make(&n.comp[i]);
  }
  if (!ok) {
    cudaGetLastError();
    for (cudaEvent_t e : made) cudaEventDestroy(e);
    if (aux_made) cudaStreamDestroy(n.aux);
    cudaGetLastError();
    return nullptr;
  }
  n.ok = true;
  h = n;
  return &h;
}

dit_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DIT_OK;
  cudaGetLastError();
  return DIT_E_CUDA;
}

// Launch the attention kernel over prepared operands.
dit_status run_attention(const void* q, const void* k, const void* v, void* out, CUtensorMapDataType qk_dt,
                         int qk_esize, int qk_format, int pv_format, int B, int Hq, int Hkv, int Sq, int Skv,
                         int mode, int q_block, int k_block, float factor, const float* q_scale,
                         const float* k_scale, const float* v_scale, int32_t* skip_counts, float* lse,
                         int* err, cudaStream_t stream, int q_hstride = 0, int kv_hstride = 0,
                         const uint8_t* q_sf = nullptr, const uint8_t* k_sf = nullptr,
                         const float* q_gs = nullptr, const float* k_gs = nullptr,
                         unsigned long long wait_budget_ns = kWaitBudgetNs, int withhold_loads = 0) {
  // q_hstride / kv_hstride: head counts of the full tensors' rows when q, k, v, out are head slices
  if (q_hstride == 0) q_hstride = Hq;
  if (kv_hstride == 0) kv_hstride = Hkv;
  CUtensorMap tq, tk, tv, to;
  const CUtensorMapDataType pv_dt =
      (pv_format == PV_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int pv_esize = (pv_format == PV_BF16) ? 2 : 1;
  const bool packed4 = (qk_format == QK_NVF4);
  if (!encode_map(&tq, q, qk_dt, qk_esize, B, Sq, Hq, q_hstride, packed4) ||
      !encode_map(&tk, k, qk_dt, qk_esize, B, Skv, Hkv, kv_hstride, packed4) ||
      !encode_map(&tv, v, pv_dt, pv_esize, B, Skv, Hkv, kv_hstride) ||
      !encode_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, Sq, Hq, q_hstride))
    return DIT_E_CUDA;
  FmhaParams p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv;
  p.group = Hq / Hkv;
  p.n_q_tiles = ceil_div(Sq, kTile);
  p.n_kv_tiles = ceil_div(Skv, kTile);
  p.c_scale = (float)(1.4426950408889634 / std::sqrt(128.0));  // softmax scale * log2(e)
  // Skip-Softmax with factor 0 (the threshold 0, the setting of the steps where skipping is off) can skip
  // nothing: it runs the kernel without the skip test, which gives the same output and LSE and writes
  // zero skip counts.
  const bool skip = (mode & DIT_MODE_SKIP) != 0 && factor > 0.0f;
  p.log2_thr = skip ? (float)std::log2((double)factor / (double)Skv) : -INFINITY;
  p.q_scale = q_scale; p.q_block = q_block; p.nqb = ceil_div(Sq, q_block);
  p.k_scale = k_scale; p.k_block = k_block; p.nkb = ceil_div(Skv, k_block);
  p.v_scale = v_scale;
  p.q_sf = q_sf;
  p.k_sf = k_sf;
  p.q_gs = q_gs;
  p.k_gs = k_gs;
  p.skip_counts = skip_counts;
  p.lse = lse;
  p.err = err;
  p.wait_budget_ns = wait_budget_ns;
  if (withhold_loads) return from_cuda(launch_fmha_withheld(pv_format, tq, tk, tv, to, p, stream));
  return from_cuda(launch_fmha(qk_format, pv_format, skip, tq, tk, tv, to, p, stream));
}

// Group boundaries for dit_attn_fwd_host: group c holds kv heads [bounds[c], bounds[c + 1]). Only the
// first group's input copies and the last group's output copy have no kernel to hide behind, so with
// five or more groups and enough kv heads the groups ramp up as 1, 2 and 4 kv heads (each group's
// inputs arrive while the one before computes: the host link moves a head's Q, K and V several times
// faster than the kernel consumes it), the middle groups split the rest evenly and the last group holds
// one kv head. Otherwise the groups are (nearly) equal.
void host_chunk_bounds(int Hkv, int chunks, int* bounds) {
  if (chunks >= 5 && Hkv - 8 >= chunks - 4) {
    const int mid = chunks - 4, rest = Hkv - 8;  // groups 3 .. chunks - 2 share heads [7, Hkv - 1)
    bounds[0] = 0;
    bounds[1] = 1;
    bounds[2] = 3;
    for (int c = 0; c <= mid; ++c) bounds[3 + c] = 7 + (int)((long long)rest * c / mid);
    bounds[chunks] = Hkv;
  } else {
    for (int c = 0; c <= chunks; ++c) bounds[c] = (int)((long long)Hkv * c / chunks);
  }
}

// The device address of the host range [p, p + bytes) when all of it is page-locked host memory mapped
// for the current device (both ends are, with device addresses bytes - 1 apart) and 16-byte aligned;
// nullptr otherwise (pageable memory, another device's mapping), in which case the caller keeps the
// copy engines.
void* pinned_device_view(const void* p, size_t bytes) {
  if (p == nullptr || bytes == 0 || !aligned16(p)) return nullptr;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  cudaPointerAttributes a{}, z{};
  const void* last = static_cast<const uint8_t*>(p) + (bytes - 1);
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess || cudaPointerGetAttributes(&z, last) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || z.type != cudaMemoryTypeHost || a.device != dev || z.device != dev ||
      a.devicePointer == nullptr || z.devicePointer == nullptr)
    return nullptr;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(a.devicePointer), d1 = reinterpret_cast<uintptr_t>(z.devicePointer);
  if (d1 < d0 || d1 - d0 != bytes - 1 || (d0 & 15u) != 0) return nullptr;
  return a.devicePointer;
}

}  // namespace

namespace ditattn {

bool is_block(int x) { return x == 1 || x == 4 || x == 16; }

// Shapes shared by every entry point. Empty problems (B == 0 or Sq == 0) are valid no-ops.
bool valid_shape(int B, int Hq, int Hkv, int Sq, int Skv) {
  if (B < 0 || Sq < 0 || Hq < 1 || Hkv < 1 || Skv < 1) return false;
  if (Hq % Hkv != 0) return false;
  if (Hq > 65535 || B > 65535) return false;  // grid y / z limits
  // every element index must fit the 64-bit offsets and TMA's 2^40-byte stride limit
  const double q_bytes = (double)B * Sq * Hq * kHeadDim * 2.0;
  const double kv_bytes = (double)B * Skv * Hkv * kHeadDim * 2.0;
  return q_bytes < 1e12 && kv_bytes < 1e12;
}

bool valid_mode(int mode, int qk_dtype, int q_block, int k_block, float factor) {
  if (mode < 0 || mode > (DIT_MODE_SAGE | DIT_MODE_SKIP | DIT_MODE_V_PER_TENSOR)) return false;
  if (mode & DIT_MODE_SAGE) {
    if (qk_dtype == DIT_QK_BF16 || qk_dtype == DIT_QK_MXFP8 || qk_dtype == DIT_QK_NVFP4) {
      // QK16PV8: Q/K stay BF16; MXFP8 / NVFP4: Q/K carry their own blocks of 32 / 16 channels. Either way
      // the token-block sizes are 0 (the pages' block sizes (0, 0, v)); V per channel or per tensor.
      if (q_block != 0 || k_block != 0) return false;
    } else {
      if (qk_dtype != DIT_QK_INT8 && qk_dtype != DIT_QK_FP8_E4M3) return false;
      if (!is_block(q_block) || !is_block(k_block)) return false;
      if (mode & DIT_MODE_V_PER_TENSOR) return false;  // the SAGE recipes scale V per channel
    }
  } else {
    if (qk_dtype != DIT_QK_BF16) return false;       // a quantized dtype without SAGE is contradictory
    if (mode & DIT_MODE_V_PER_TENSOR) return false;  // V is not quantized without SAGE
  }
  if (mode & DIT_MODE_SKIP) {
    if (!std::isfinite(factor) || factor < 0.0f) return false;
  }
  return true;
}

}  // namespace ditattn

extern "C" {

int dit_abi_version(void) { return kAbiVersion; }

const char* dit_status_string(dit_status s) {
  switch (s) {
    case DIT_OK: return "ok";
    case DIT_E_INVALID_ARG: return "invalid argument";
    case DIT_E_UNSUPPORTED: return "unsupported device (needs an sm_103 GPU)";
    case DIT_E_CUDA: return "CUDA error";
    case DIT_E_TIMEOUT: return "kernel wait timed out";
    case DIT_E_WORKSPACE: return "workspace missing or too small";
    case DIT_E_BOUNDS: return "index outside its buffer (bounds-checked build)";
  }
  return "unknown status";
}

size_t dit_attn_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int mode, int qk_dtype, int q_block,
                                int k_block) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || !valid_mode(mode, qk_dtype, q_block, k_block, 0.0f)) return 0;
  if (!(mode & DIT_MODE_SAGE)) return 0;
  return sage_layout(B, Hq, Hkv, Sq, Skv, qk_dtype, q_block, k_block).total;
}

}  // extern "C"

namespace {

// dit_attn_fwd and dit_attn_fwd_lse (lse may be NULL).
dit_status fwd_impl(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv, int Sq, int Skv,
                    int mode, int qk_dtype, int q_block, int k_block, float threshold_scale_factor, void* stream,
                    void* workspace, size_t workspace_bytes, int32_t* skip_counts, float* lse) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || !valid_mode(mode, qk_dtype, q_block, k_block, threshold_scale_factor))
    return DIT_E_INVALID_ARG;
  if (B == 0 || Sq == 0) return DIT_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(skip_counts) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DIT_E_INVALID_ARG;
  const bool sage = (mode & DIT_MODE_SAGE) != 0;
  SageLayout L{};
  if (sage) {
    L = sage_layout(B, Hq, Hkv, Sq, Skv, qk_dtype, q_block, k_block);
    if (workspace == nullptr || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return DIT_E_WORKSPACE;
  }
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!sage)
    return run_attention(q, k, v, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, QK_BF16, PV_BF16, B, Hq, Hkv, Sq, Skv,
                         mode, 1, 1, threshold_scale_factor, nullptr, nullptr, nullptr, skip_counts, lse, err, st);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (qk_dtype == DIT_QK_NVFP4) {
    // NVFP4 Q/K + FP8 V: V as in QK16PV8; Q/K codes, block scales and the two tensor scales
    float* v_scale = reinterpret_cast<float*>(ws + L.v_scale);
    float* gs = reinterpret_cast<float*>(ws + L.gs);
    cudaError_t e = launch_v_stats(v, B, Hkv, Skv, reinterpret_cast<float*>(ws + L.pmax), v_scale,
                                   (mode & DIT_MODE_V_PER_TENSOR) != 0, st);
    if (e == cudaSuccess) e = launch_quant_v(v, B, Hkv, Skv, v_scale, ws + L.v_codes, st);
    if (e == cudaSuccess)
      e = launch_nvfp4_quant(q, k, B, Hq, Hkv, Sq, Skv, ws + L.q_codes, ws + L.k_codes, ws + L.q_scale,
                             ws + L.k_scale, gs, gs + 1, st);
    if (e != cudaSuccess) return from_cuda(e);
    return run_attention(ws + L.q_codes, ws + L.k_codes, ws + L.v_codes, out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                         QK_NVF4, PV_E4M3, B, Hq, Hkv, Sq, Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr,
                         v_scale, skip_counts, lse, err, st, 0, 0, ws + L.q_scale, ws + L.k_scale, gs, gs + 1);
  }
  if (qk_dtype == DIT_QK_MXFP8) {
    // MXFP8 Q/K + FP8 V: V scales and codes as in QK16PV8, Q/K codes with their E8M0 block scales
    float* v_scale = reinterpret_cast<float*>(ws + L.v_scale);
    uint8_t* q_sf = ws + L.q_scale;
    uint8_t* k_sf = ws + L.k_scale;
    cudaError_t e = launch_v_stats(v, B, Hkv, Skv, reinterpret_cast<float*>(ws + L.pmax), v_scale,
                                   (mode & DIT_MODE_V_PER_TENSOR) != 0, st);
    if (e == cudaSuccess) e = launch_quant_v(v, B, Hkv, Skv, v_scale, ws + L.v_codes, st);
    if (e == cudaSuccess) e = launch_mx_quant(q, B, Sq, Hq, ws + L.q_codes, q_sf, st);
    if (e == cudaSuccess) e = launch_mx_quant(k, B, Skv, Hkv, ws + L.k_codes, k_sf, st);
    if (e != cudaSuccess) return from_cuda(e);
    return run_attention(ws + L.q_codes, ws + L.k_codes, ws + L.v_codes, out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                         QK_MXF8, PV_E4M3, B, Hq, Hkv, Sq, Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr,
                         v_scale, skip_counts, lse, err, st, 0, 0, q_sf, k_sf);
  }
  if (qk_dtype == DIT_QK_BF16) {
    // QK16PV8: V scales (per channel or one tensor-wide) and V codes; Q/K go to BMM1 as they are
    float* v_scale = reinterpret_cast<float*>(ws + L.v_scale);
    cudaError_t e = launch_v_stats(v, B, Hkv, Skv, reinterpret_cast<float*>(ws + L.pmax), v_scale,
                                   (mode & DIT_MODE_V_PER_TENSOR) != 0, st);
    if (e == cudaSuccess) e = launch_quant_v(v, B, Hkv, Skv, v_scale, ws + L.v_codes, st);
    if (e != cudaSuccess) return from_cuda(e);
    return run_attention(q, k, ws + L.v_codes, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, QK_BF16, PV_E4M3, B, Hq,
                         Hkv, Sq, Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr, v_scale, skip_counts,
                         lse, err, st);
  }
  float* q_scale = reinterpret_cast<float*>(ws + L.q_scale);
  float* k_scale = reinterpret_cast<float*>(ws + L.k_scale);
  float* v_scale = reinterpret_cast<float*>(ws + L.v_scale);
  float* k_mean = reinterpret_cast<float*>(ws + L.k_mean);
  const int code_out = (qk_dtype == DIT_QK_INT8) ? CODE_I8_AS_F16 : CODE_E4M3;
  cudaError_t e = launch_kv_stats(k, v, B, Hkv, Skv, reinterpret_cast<double*>(ws + L.psum),
                                  reinterpret_cast<float*>(ws + L.pmax), k_mean, v_scale, st);
  if (e == cudaSuccess) e = launch_quant_q(q, B, Hq, Sq, q_block, code_out, ws + L.q_codes, q_scale, st, true);
  if (e == cudaSuccess)
    e = launch_quant_kv(k, v, B, Hkv, Skv, k_block, code_out, k_mean, v_scale, ws + L.k_codes, k_scale,
                        ws + L.v_codes, st);
  if (e != cudaSuccess) return from_cuda(e);
  const bool i8 = (qk_dtype == DIT_QK_INT8);
  return run_attention(ws + L.q_codes, ws + L.k_codes, ws + L.v_codes, out,
                       i8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, i8 ? 2 : 1,
                       i8 ? QK_F16 : QK_E4M3, PV_E4M3, B, Hq, Hkv, Sq, Skv, mode, q_block, k_block,
                       threshold_scale_factor, q_scale, k_scale, v_scale, skip_counts, lse, err, st);
}

}  // namespace

extern "C" {

dit_status dit_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv, int Sq,
                        int Skv, int mode, int qk_dtype, int q_block, int k_block, float threshold_scale_factor,
                        void* stream, void* workspace, size_t workspace_bytes, int32_t* skip_counts) {
  return fwd_impl(q, k, v, out, B, Hq, Hkv, Sq, Skv, mode, qk_dtype, q_block, k_block, threshold_scale_factor, stream,
                  workspace, workspace_bytes, skip_counts, nullptr);
}

dit_status dit_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                            int Hkv, int Sq, int Skv, int mode, int qk_dtype, int q_block, int k_block,
                            float threshold_scale_factor, void* stream, void* workspace, size_t workspace_bytes,
                            int32_t* skip_counts) {
  if (lse == nullptr) return DIT_E_INVALID_ARG;
  return fwd_impl(q, k, v, out, B, Hq, Hkv, Sq, Skv, mode, qk_dtype, q_block, k_block, threshold_scale_factor, stream,
                  workspace, workspace_bytes, skip_counts, lse);
}

size_t sage_quantize_workspace_bytes(int B, int Hkv, int Skv) {
  if (B < 0 || Hkv < 1 || Skv < 1) return 0;
  return stats_bytes(B, Hkv, Skv);
}

dit_status sage_quantize_qkv(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Sq, int Skv,
                             int qk_dtype, int q_block, int k_block, void* q_codes, void* k_codes, void* v_codes,
                             float* q_scale, float* k_scale, float* v_scale, float* k_mean, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || (qk_dtype != DIT_QK_INT8 && qk_dtype != DIT_QK_FP8_E4M3) ||
      !valid_mode(DIT_MODE_SAGE, qk_dtype, q_block, k_block, 0.0f))
    return DIT_E_INVALID_ARG;
  if (B == 0) return DIT_OK;
  const void* ptrs[] = {k, v, k_codes, v_codes, k_scale, v_scale, k_mean};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return DIT_E_INVALID_ARG;
  if (Sq > 0 && (!q || !q_codes || !q_scale || !aligned16(q) || !aligned16(q_codes))) return DIT_E_INVALID_ARG;
  const size_t need = stats_bytes(B, Hkv, Skv);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DIT_E_WORKSPACE;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t n = (size_t)B * Hkv * stats_chunks(Skv) * kHeadDim;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int code_out = (qk_dtype == DIT_QK_INT8) ? CODE_I8 : CODE_E4M3;
  cudaError_t e = launch_kv_stats(k, v, B, Hkv, Skv, reinterpret_cast<double*>(ws),
                                  reinterpret_cast<float*>(ws + align256(n * 8)), k_mean, v_scale, st);
  if (e == cudaSuccess && Sq > 0) e = launch_quant_q(q, B, Hq, Sq, q_block, code_out, q_codes, q_scale, st, true);
  if (e == cudaSuccess)
    e = launch_quant_kv(k, v, B, Hkv, Skv, k_block, code_out, k_mean, v_scale, k_codes, k_scale, v_codes, st);
  return from_cuda(e);
}

dit_status sage_quantize_qkv_with_mean(const void* q, const void* k, const void* v, const float* k_mean, int B,
                                       int Hq, int Hkv, int Sq, int Skv, int qk_dtype, int q_block, int k_block,
                                       void* q_codes, void* k_codes, void* v_codes, float* q_scale, float* k_scale,
                                       float* v_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || (qk_dtype != DIT_QK_INT8 && qk_dtype != DIT_QK_FP8_E4M3) ||
      !valid_mode(DIT_MODE_SAGE, qk_dtype, q_block, k_block, 0.0f))
    return DIT_E_INVALID_ARG;
  if (B == 0) return DIT_OK;
  const void* ptrs[] = {k, v, k_mean, k_codes, v_codes, k_scale, v_scale};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return DIT_E_INVALID_ARG;
  if (Sq > 0 && (!q || !q_codes || !q_scale || !aligned16(q) || !aligned16(q_codes))) return DIT_E_INVALID_ARG;
  const size_t need = align256((size_t)B * Hkv * stats_chunks(Skv) * kHeadDim * 4);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DIT_E_WORKSPACE;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int code_out = (qk_dtype == DIT_QK_INT8) ? CODE_I8 : CODE_E4M3;
  cudaError_t e = launch_v_stats(v, B, Hkv, Skv, static_cast<float*>(workspace), v_scale, false, st);
  if (e == cudaSuccess && Sq > 0) e = launch_quant_q(q, B, Hq, Sq, q_block, code_out, q_codes, q_scale, st);
  if (e == cudaSuccess)
    e = launch_quant_kv(k, v, B, Hkv, Skv, k_block, code_out, k_mean, v_scale, k_codes, k_scale, v_codes, st);
  return from_cuda(e);
}

size_t sage_quantize_v_workspace_bytes(int B, int Hkv, int Skv) {
  if (B < 0 || Hkv < 1 || Skv < 1) return 0;
  return align256((size_t)B * Hkv * stats_chunks(Skv) * kHeadDim * 4);
}

dit_status sage_quantize_v(const void* v, int B, int Hkv, int Skv, int v_per_tensor, void* v_codes, float* v_scale,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_shape(B, Hkv, Hkv, 0, Skv) || (v_per_tensor != 0 && v_per_tensor != 1)) return DIT_E_INVALID_ARG;
  if (B == 0) return DIT_OK;
  if (!v || !v_codes || !v_scale || !aligned16(v) || !aligned16(v_codes) || !aligned16(v_scale))
    return DIT_E_INVALID_ARG;
  const size_t need = sage_quantize_v_workspace_bytes(B, Hkv, Skv);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DIT_E_WORKSPACE;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_v_stats(v, B, Hkv, Skv, static_cast<float*>(workspace), v_scale, v_per_tensor != 0, st);
  if (e == cudaSuccess) e = launch_quant_v(v, B, Hkv, Skv, v_scale, v_codes, st);
  return from_cuda(e);
}

size_t dit_attn_quantized_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int qk_dtype) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv)) return 0;
  if (qk_dtype == DIT_QK_FP8_E4M3) return 0;
  if (qk_dtype != DIT_QK_INT8) return 0;
  return align256((size_t)B * Sq * Hq * kHeadDim * 2) + align256((size_t)B * Skv * Hkv * kHeadDim * 2);
}

}  // extern "C"

namespace {

// dit_attn_fwd_quantized and dit_attn_fwd_quantized_lse (lse may be NULL).
dit_status fwd_quantized_impl(const void* q_codes, const void* k_codes, const void* v_codes, const float* q_scale,
                              const float* k_scale, const float* v_scale, void* out, int B, int Hq, int Hkv, int Sq,
                              int Skv, int mode, int qk_dtype, int q_block, int k_block, float threshold_scale_factor,
                              void* stream, void* workspace, size_t workspace_bytes, int32_t* skip_counts,
                              float* lse) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || !(mode & DIT_MODE_SAGE) || qk_dtype == DIT_QK_MXFP8 ||
      qk_dtype == DIT_QK_NVFP4 || !valid_mode(mode, qk_dtype, q_block, k_block, threshold_scale_factor))
    return DIT_E_INVALID_ARG;  // MXFP8 / NVFP4 operands go through dit_attn_fwd_mxfp8 / dit_attn_fwd_nvfp4
  if (B == 0 || Sq == 0) return DIT_OK;
  const bool qk16 = (qk_dtype == DIT_QK_BF16);  // QK16PV8: q_codes / k_codes are the BF16 Q / K, no Q/K scales
  const void* ptrs[] = {q_codes, k_codes, v_codes, v_scale, out};
  for (const void* ptr : ptrs)
    if (!ptr) return DIT_E_INVALID_ARG;
  if (!qk16 && (!q_scale || !k_scale)) return DIT_E_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(out) ||
      !aligned16(skip_counts) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DIT_E_INVALID_ARG;
  const bool i8 = (qk_dtype == DIT_QK_INT8);
  const size_t need = dit_attn_quantized_workspace_bytes(B, Hq, Hkv, Sq, Skv, qk_dtype);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return DIT_E_WORKSPACE;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* qa = q_codes;
  const void* ka = k_codes;
  if (i8) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t nq = (size_t)B * Sq * Hq * kHeadDim, nk = (size_t)B * Skv * Hkv * kHeadDim;
    void* q16 = ws;
    void* k16 = ws + align256(nq * 2);
    cudaError_t e = launch_widen_i8(static_cast<const int8_t*>(q_codes), nq, q16, st);
    if (e == cudaSuccess) e = launch_widen_i8(static_cast<const int8_t*>(k_codes), nk, k16, st);
    if (e != cudaSuccess) return from_cuda(e);
    qa = q16;
    ka = k16;
  }
  if (qk16)
    return run_attention(qa, ka, v_codes, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, QK_BF16, PV_E4M3, B, Hq, Hkv, Sq,
                         Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr, v_scale, skip_counts, lse, err, st);
  return run_attention(qa, ka, v_codes, out, i8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                       i8 ? 2 : 1, i8 ? QK_F16 : QK_E4M3, PV_E4M3, B, Hq, Hkv, Sq, Skv, mode, q_block, k_block,
                       threshold_scale_factor, q_scale, k_scale, v_scale, skip_counts, lse, err, st);
}

}  // namespace

extern "C" {

dit_status dit_attn_fwd_quantized(const void* q_codes, const void* k_codes, const void* v_codes,
                                  const float* q_scale, const float* k_scale, const float* v_scale, void* out, int B,
                                  int Hq, int Hkv, int Sq, int Skv, int mode, int qk_dtype, int q_block, int k_block,
                                  float threshold_scale_factor, void* stream, void* workspace,
                                  size_t workspace_bytes, int32_t* skip_counts) {
  return fwd_quantized_impl(q_codes, k_codes, v_codes, q_scale, k_scale, v_scale, out, B, Hq, Hkv, Sq, Skv, mode,
                            qk_dtype, q_block, k_block, threshold_scale_factor, stream, workspace, workspace_bytes,
                            skip_counts, nullptr);
}

dit_status dit_attn_fwd_quantized_lse(const void* q_codes, const void* k_codes, const void* v_codes,
                                      const float* q_scale, const float* k_scale, const float* v_scale, void* out,
                                      float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int mode, int qk_dtype,
                                      int q_block, int k_block, float threshold_scale_factor, void* stream,
                                      void* workspace, size_t workspace_bytes, int32_t* skip_counts) {
  if (lse == nullptr) return DIT_E_INVALID_ARG;
  return fwd_quantized_impl(q_codes, k_codes, v_codes, q_scale, k_scale, v_scale, out, B, Hq, Hkv, Sq, Skv, mode,
                            qk_dtype, q_block, k_block, threshold_scale_factor, stream, workspace, workspace_bytes,
                            skip_counts, lse);
}

dit_status mx_quantize_qk(const void* q, const void* k, int B, int Hq, int Hkv, int Sq, int Skv, void* q_codes,
                          void* k_codes, uint8_t* q_sf, uint8_t* k_sf, void* stream) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv)) return DIT_E_INVALID_ARG;
  if (B == 0) return DIT_OK;
  if (!k || !k_codes || !k_sf || !aligned16(k) || !aligned16(k_codes) || (reinterpret_cast<uintptr_t>(k_sf) & 3u))
    return DIT_E_INVALID_ARG;
  if (Sq > 0 && (!q || !q_codes || !q_sf || !aligned16(q) || !aligned16(q_codes) ||
                 (reinterpret_cast<uintptr_t>(q_sf) & 3u)))
    return DIT_E_INVALID_ARG;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (Sq > 0) e = launch_mx_quant(q, B, Sq, Hq, q_codes, q_sf, st);
  if (e == cudaSuccess) e = launch_mx_quant(k, B, Skv, Hkv, k_codes, k_sf, st);
  return from_cuda(e);
}

dit_status dit_attn_fwd_mxfp8(const void* q_codes, const void* k_codes, const void* v_codes, const uint8_t* q_sf,
                              const uint8_t* k_sf, const float* v_scale, void* out, float* lse, int B, int Hq,
                              int Hkv, int Sq, int Skv, int mode, float threshold_scale_factor, void* stream,
                              int32_t* skip_counts) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || !(mode & DIT_MODE_SAGE) ||
      !valid_mode(mode, DIT_QK_MXFP8, 0, 0, threshold_scale_factor))
    return DIT_E_INVALID_ARG;
  if (B == 0 || Sq == 0) return DIT_OK;
  const void* ptrs[] = {q_codes, k_codes, v_codes, q_sf, k_sf, v_scale, out};
  for (const void* ptr : ptrs)
    if (!ptr) return DIT_E_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(out) ||
      !aligned16(skip_counts) || (reinterpret_cast<uintptr_t>(q_sf) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_sf) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DIT_E_INVALID_ARG;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  return run_attention(q_codes, k_codes, v_codes, out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, QK_MXF8, PV_E4M3, B, Hq,
                       Hkv, Sq, Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr, v_scale, skip_counts, lse,
                       err, static_cast<cudaStream_t>(stream), 0, 0, q_sf, k_sf);
}

dit_status nvfp4_quantize_qk(const void* q, const void* k, int B, int Hq, int Hkv, int Sq, int Skv, void* q_codes,
                            void* k_codes, uint8_t* q_sf, uint8_t* k_sf, float* q_scale, float* k_scale,
                            void* stream) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv)) return DIT_E_INVALID_ARG;
  if (B == 0) return DIT_OK;
  if (!k || !k_codes || !k_sf || !k_scale || !aligned16(k) || !aligned16(k_codes) ||
      (reinterpret_cast<uintptr_t>(k_sf) & 7u) || (reinterpret_cast<uintptr_t>(k_scale) & 3u))
    return DIT_E_INVALID_ARG;
  if (Sq > 0 && (!q || !q_codes || !q_sf || !q_scale || !aligned16(q) || !aligned16(q_codes) ||
                 (reinterpret_cast<uintptr_t>(q_sf) & 7u) || (reinterpret_cast<uintptr_t>(q_scale) & 3u)))
    return DIT_E_INVALID_ARG;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  return from_cuda(launch_nvfp4_quant(Sq > 0 ? q : nullptr, k, B, Hq, Hkv, Sq, Skv, q_codes, k_codes, q_sf, k_sf,
                                      q_scale, k_scale, static_cast<cudaStream_t>(stream)));
}

dit_status dit_attn_fwd_nvfp4(const void* q_codes, const void* k_codes, const void* v_codes, const uint8_t* q_sf,
                              const uint8_t* k_sf, const float* q_scale, const float* k_scale, const float* v_scale,
                              void* out, float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int mode,
                              float threshold_scale_factor, void* stream, int32_t* skip_counts) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || !(mode & DIT_MODE_SAGE) ||
      !valid_mode(mode, DIT_QK_NVFP4, 0, 0, threshold_scale_factor))
    return DIT_E_INVALID_ARG;
  if (B == 0 || Sq == 0) return DIT_OK;
  const void* ptrs[] = {q_codes, k_codes, v_codes, q_sf, k_sf, q_scale, k_scale, v_scale, out};
  for (const void* ptr : ptrs)
    if (!ptr) return DIT_E_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(out) ||
      !aligned16(skip_counts) || (reinterpret_cast<uintptr_t>(q_sf) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_sf) & 7u) || (reinterpret_cast<uintptr_t>(q_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DIT_E_INVALID_ARG;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  return run_attention(q_codes, k_codes, v_codes, out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, QK_NVF4, PV_E4M3, B, Hq,
                       Hkv, Sq, Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr, v_scale, skip_counts, lse,
                       err, static_cast<cudaStream_t>(stream), 0, 0, q_sf, k_sf, q_scale, k_scale);
}

dit_status dit_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* out_host, void* q,
                             void* k, void* v, void* out, int B, int Hq, int Hkv, int Sq, int Skv, int mode,
                             float threshold_scale_factor, int chunks, void* compute_stream, void* h2d_stream,
                             void* d2h_stream) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || (mode & ~DIT_MODE_SKIP) != 0 ||
      !valid_mode(mode, DIT_QK_BF16, 1, 1, threshold_scale_factor) || chunks < 1 || chunks > Hkv ||
      chunks > kMaxHostChunks)
    return DIT_E_INVALID_ARG;
  if (B == 0 || Sq == 0) return DIT_OK;
  if (!q_host || !k_host || !v_host || !out_host || !q || !k || !v || !out || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(out))
    return DIT_E_INVALID_ARG;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  HostEvents* ev = host_events();
  if (ev == nullptr) return DIT_E_CUDA;
  std::lock_guard<std::mutex> call_lock(g_host_call_mu);
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t hs = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ds2 = static_cast<cudaStream_t>(d2h_stream);
  const int group = Hq / Hkv;
  const size_t row = (size_t)kHeadDim * 2;  // bytes of one head of one token
  // the copies may not overwrite the device buffers before earlier work on the compute stream is done
  cudaError_t e = cudaEventRecord(ev->start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs, ev->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds2, ev->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ev->aux, ev->start, 0);
  // chunk c covers kv heads [bounds[c], bounds[c + 1]) and their query heads
  int bounds[kMaxHostChunks + 1];
  host_chunk_bounds(Hkv, chunks, bounds);
  auto kv0 = [&](int c) { return bounds[c]; };
  // The first group's inputs and the last group's output are copied by SM kernels when the host
  // buffers are page-locked (no attention kernel runs at those times); everything else by the copy
  // engines, overlapped with the attention.
  const size_t q_bytes = (size_t)B * Sq * Hq * row, kv_bytes = (size_t)B * Skv * Hkv * row;
  const void* qh_dev = pinned_device_view(q_host, q_bytes);
  const void* kh_dev = pinned_device_view(k_host, kv_bytes);
  const void* vh_dev = pinned_device_view(v_host, kv_bytes);
  void* oh_dev = pinned_device_view(out_host, q_bytes);
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int hk0 = kv0(c), hkc = kv0(c + 1) - hk0, hq0 = hk0 * group, hqc = hkc * group;
    const size_t qo = hq0 * row, ko = hk0 * row;
    if (c == 0 && qh_dev != nullptr && kh_dev != nullptr && vh_dev != nullptr) {
      e = launch_copy_rows(static_cast<const uint8_t*>(qh_dev) + qo, Hq * row, static_cast<uint8_t*>(q) + qo, Hq * row,
                           hqc * row, (size_t)B * Sq, hs);
      if (e == cudaSuccess)
        e = launch_copy_rows(static_cast<const uint8_t*>(kh_dev) + ko, Hkv * row, static_cast<uint8_t*>(k) + ko,
                             Hkv * row, hkc * row, (size_t)B * Skv, hs);
      if (e == cudaSuccess)
        e = launch_copy_rows(static_cast<const uint8_t*>(vh_dev) + ko, Hkv * row, static_cast<uint8_t*>(v) + ko,
                             Hkv * row, hkc * row, (size_t)B * Skv, hs);
    } else {
      e = cudaMemcpy2DAsync(static_cast<uint8_t*>(q) + qo, Hq * row, static_cast<const uint8_t*>(q_host) + qo,
                            Hq * row, hqc * row, (size_t)B * Sq, cudaMemcpyHostToDevice, hs);
      if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(static_cast<uint8_t*>(k) + ko, Hkv * row, static_cast<const uint8_t*>(k_host) + ko,
                              Hkv * row, hkc * row, (size_t)B * Skv, cudaMemcpyHostToDevice, hs);
      if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(static_cast<uint8_t*>(v) + ko, Hkv * row, static_cast<const uint8_t*>(v_host) + ko,
                              Hkv * row, hkc * row, (size_t)B * Skv, cudaMemcpyHostToDevice, hs);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev->in[c], hs);
  }
  dit_status failed = DIT_OK;  // a group's launch that failed (its copies are still joined below)
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int hk0 = kv0(c), hkc = kv0(c + 1) - hk0, hq0 = hk0 * group, hqc = hkc * group;
    cudaStream_t ks = (c & 1) ? ev->aux : cs;
    e = cudaStreamWaitEvent(ks, ev->in[c], 0);
    if (e != cudaSuccess) break;
    const dit_status st = run_attention(
        static_cast<uint8_t*>(q) + hq0 * row, static_cast<uint8_t*>(k) + hk0 * row,
        static_cast<uint8_t*>(v) + hk0 * row, static_cast<uint8_t*>(out) + hq0 * row, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
        2, QK_BF16, PV_BF16, B, hqc, hkc, Sq, Skv, mode, 1, 1, threshold_scale_factor, nullptr, nullptr, nullptr,
        nullptr, nullptr, err, ks, Hq, Hkv);
    if (st != DIT_OK) {
      failed = st;
      break;
    }
    e = cudaEventRecord(ev->comp[c], ks);
  }
  // On a failure nothing more is queued. The copies and kernels already queued on the copy streams
  // and on `aux` are joined back to the compute stream, so that once it drains the caller may reuse
  // or free every buffer; if even that cannot be queued, this waits for them.
  auto fail_joined = [&](dit_status ret) {
    cudaGetLastError();
    const bool joined = cudaEventRecord(ev->h2d_done, hs) == cudaSuccess &&
                        cudaEventRecord(ev->done, ds2) == cudaSuccess &&
                        cudaEventRecord(ev->aux_done, ev->aux) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, ev->h2d_done, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, ev->done, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, ev->aux_done, 0) == cudaSuccess;
    if (!joined) {
      cudaGetLastError();
      cudaStreamSynchronize(hs);
      cudaStreamSynchronize(ds2);
      cudaStreamSynchronize(ev->aux);
      cudaGetLastError();
    }
    return ret;
  };
  if (failed != DIT_OK) return fail_joined(failed);
  if (e != cudaSuccess) return fail_joined(DIT_E_CUDA);
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int hk0 = kv0(c), hkc = kv0(c + 1) - hk0, hq0 = hk0 * group, hqc = hkc * group;
    const size_t qo = hq0 * row;
    e = cudaStreamWaitEvent(ds2, ev->comp[c], 0);
    if (e != cudaSuccess) break;
    if (c == chunks - 1 && oh_dev != nullptr) {
      // d2h_stream has waited for every group's kernel by now, so no attention kernel is running
      e = launch_copy_rows(static_cast<const uint8_t*>(out) + qo, Hq * row, static_cast<uint8_t*>(oh_dev) + qo, Hq * row,
                           hqc * row, (size_t)B * Sq, ds2);
    } else {
      e = cudaMemcpy2DAsync(static_cast<uint8_t*>(out_host) + qo, Hq * row, static_cast<const uint8_t*>(out) + qo,
                            Hq * row, hqc * row, (size_t)B * Sq, cudaMemcpyDeviceToHost, ds2);
    }
  }
  if (e != cudaSuccess) return fail_joined(DIT_E_CUDA);
  // completion (the last output byte on the host, and all kernels) is signalled on the compute stream
  e = cudaEventRecord(ev->done, ds2);
  if (e == cudaSuccess) e = cudaEventRecord(ev->aux_done, ev->aux);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev->done, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev->aux_done, 0);
  if (e != cudaSuccess) return fail_joined(DIT_E_CUDA);
  return DIT_OK;
}

dit_status dit_selftest_withheld_loads(const void* q, const void* k, const void* v, const float* v_scale, void* out,
                                      int B, int Hq, int Hkv, int Sq, int Skv, int e4m3_v,
                                      unsigned long long wait_budget_ns, void* stream) {
  if (!valid_shape(B, Hq, Hkv, Sq, Skv) || B == 0 || Sq == 0 || (e4m3_v != 0 && e4m3_v != 1) ||
      wait_budget_ns < 1000000ull || wait_budget_ns > 10000000000ull)
    return DIT_E_INVALID_ARG;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (e4m3_v && !v_scale))
    return DIT_E_INVALID_ARG;
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  return run_attention(q, k, v, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, QK_BF16, e4m3_v ? PV_E4M3 : PV_BF16, B, Hq,
                       Hkv, Sq, Skv, e4m3_v ? DIT_MODE_SAGE : DIT_MODE_DENSE, 1, 1, 0.0f, nullptr, nullptr,
                       e4m3_v ? v_scale : nullptr, nullptr, nullptr, err, static_cast<cudaStream_t>(stream), 0, 0,
                       nullptr, nullptr, nullptr, nullptr, wait_budget_ns, 1);
}

dit_status dit_attn_check_errors(void* stream) {
  int* err = nullptr;
  const dit_status ds = prepare_device(&err);
  if (ds != DIT_OK) return ds;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return DIT_E_CUDA;
  }
  int h = 0;
  if (cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return from_cuda(cudaErrorUnknown);
  if (h != 0) {
    const int zero = 0;
    cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return (dit_status)h;
  }
  return DIT_OK;
}

}  // extern "C"
