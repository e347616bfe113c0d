// Declarations shared by the library's translation units (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ditattn {

constexpr int kHeadDim = 128;
constexpr int kTile = 128;
constexpr int kStatsChunk = 1024;  // tokens per CTA in the K-mean / V-absmax partial pass
constexpr int kQuantRows = 256;    // tokens per CTA in the quantizers

// Storage formats of the Q/K operands of BMM1 and the V operand of BMM2.
// QK_F16: INT8 codes held exactly as fp16. QK_MXF8: E4M3 codes with E8M0 scales per 32 channels.
// QK_NVF4: E2M1 codes (two per byte) with E4M3 scales per 16 channels and a float32 tensor scale.
enum QKFormat { QK_BF16 = 0, QK_F16 = 1, QK_E4M3 = 2, QK_MXF8 = 3, QK_NVF4 = 4 };
enum PVFormat { PV_BF16 = 0, PV_E4M3 = 1 };

// Output formats of the Q/K quantizer.
enum CodeOut { CODE_I8 = 0, CODE_I8_AS_F16 = 1, CODE_E4M3 = 2 };

// Device error word codes (match dit_status).
constexpr int kErrTimeout = 4;
constexpr int kErrBounds = 6;  // DIT_E_BOUNDS: only a bounds-checked build records it

struct FmhaParams {
  int B, Hq, Hkv, Sq, Skv;
  int group;          // Hq / Hkv
  int n_q_tiles;      // ceil(Sq / 128)
  int n_kv_tiles;     // ceil(Skv / 128)
  float c_scale;      // softmax scale * log2(e)
  float log2_thr;     // log2(threshold_scale_factor / Skv); -inf when the factor is 0
  const float* q_scale;  // SAGE: [B, Hq, nqb]
  int q_block, nqb;
  const float* k_scale;  // SAGE: [B, Hkv, nkb]
  int k_block, nkb;
  const float* v_scale;  // E4M3 V (SAGE, QK16PV8, MXFP8): [B, Hkv, 128]
  const uint8_t* q_sf;   // MXFP8: E8M0 bytes [B, Hq, Sq, 4] (byte c scales channels 32c .. 32c+31)
  const uint8_t* k_sf;   // MXFP8: E8M0 bytes [B, Hkv, Skv, 4]; NVFP4: E4M3 bytes [.., 8] (16 channels each)
  const float* q_gs;     // NVFP4: the Q and K tensor scales S (BMM1 is divided by S_Q * S_K)
  const float* k_gs;
  int32_t* skip_counts;  // optional [B, Hq, n_q_tiles]
  float* lse;            // optional [B, Hq, Sq]: ln sum_j exp(s_ij) of each query row
  int* err;              // device error word
  unsigned long long wait_budget_ns;
};

// Attention kernel launcher (fmha_sm103.cu). Tensor maps describe q, k, v, out as 4-D
// {128, S, H, B} tensors with 128-byte swizzled boxes.
cudaError_t launch_fmha(int qk_format, int pv_format, bool skip, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v, const CUtensorMap& tm_o, const FmhaParams& p, cudaStream_t stream);
// The timeout-path self-test: the dense (PV_BF16) or QK16PV8 (PV_E4M3) kernel with its loads withheld.
cudaError_t launch_fmha_withheld(int pv_format, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_withheld_dense(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_withheld_qk16pv8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                         const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_dense(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_sage_i8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_sage_f8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_qk16pv8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_nvfp4(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);
cudaError_t launch_fmha_mxfp8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream);

// Quantize-prepass launchers (prepass.cu). launch_kv_stats, then launch_quant_q with after_stats
// set, then launch_quant_kv is the SAGE order: the Q quantizer then starts while the statistics are
// combined, and the V quantizer while the K quantizer's last CTAs run (programmatic dependent launch);
// each kernel in that chain still completes after the one before it, so an ordinary launch after
// launch_quant_kv sees all of their results.
cudaError_t launch_kv_stats(const void* k, const void* v, int B, int Hkv, int Skv, double* psum, float* pmax,
                            float* k_mean, float* v_scale, cudaStream_t stream);
// V alone (QK16PV8): per-channel absmax scales, optionally reduced to one tensor-wide scale
// broadcast over [B, Hkv, 128], then E4M3 codes of V / scale.
cudaError_t launch_v_stats(const void* v, int B, int Hkv, int Skv, float* pmax, float* v_scale, bool per_tensor,
                           cudaStream_t stream);
cudaError_t launch_quant_v(const void* v, int B, int Hkv, int Skv, const float* v_scale, void* v_codes,
                           cudaStream_t stream);
cudaError_t launch_quant_q(const void* q, int B, int Hq, int Sq, int q_block, int code_out, void* q_codes,
                           float* q_scale, cudaStream_t stream, bool after_stats = false);
cudaError_t launch_quant_kv(const void* k, const void* v, int B, int Hkv, int Skv, int k_block, int code_out,
                            const float* k_mean, const float* v_scale, void* k_codes, float* k_scale, void* v_codes,
                            cudaStream_t stream);
// MXFP8 codes of a [B, S, H, 128] BF16 tensor and its E8M0 scale bytes [B, H, S, 4].
cudaError_t launch_mx_quant(const void* x, int B, int S, int H, void* codes, uint8_t* sf, cudaStream_t stream);
// NVFP4 codes (packed [B, S, H, 64]), E4M3 block-scale bytes [B, H, S, 8] and the float32 tensor scales
// of Q and K (q may be skipped with Sq == 0).
cudaError_t launch_nvfp4_quant(const void* q, const void* k, int B, int Hq, int Hkv, int Sq, int Skv, void* q_codes,
                               void* k_codes, uint8_t* q_sf, uint8_t* k_sf, float* q_scale, float* k_scale,
                               cudaStream_t stream);
cudaError_t launch_widen_i8(const int8_t* codes, size_t n, void* out_f16, cudaStream_t stream);
cudaError_t launch_zero_i32(int32_t* p, size_t n, cudaStream_t stream);
// SM-driven copy of `rows` rows of `width` bytes (src/dst pitches in bytes; addresses, pitches and
// width multiples of 16); either side may be the device mapping of page-locked host memory.
cudaError_t launch_copy_rows(const void* src, size_t src_pitch, void* dst, size_t dst_pitch, size_t width,
                             size_t rows, cudaStream_t stream);

// Argument checks shared by the entry points (api.cu). valid_shape: B, Sq >= 0; Hq, Hkv, Skv >= 1;
// Hq a multiple of Hkv; grid limits; every tensor under 1e12 bytes. valid_mode: the mode bits, Q/K
// dtype and token-block sizes form a recipe the library implements, and a Skip-Softmax factor is
// finite and non-negative.
bool is_block(int x);
bool valid_shape(int B, int Hq, int Hkv, int Sq, int Skv);
bool valid_mode(int mode, int qk_dtype, int q_block, int k_block, float factor);

inline int stats_chunks(int Skv) { return (Skv + kStatsChunk - 1) / kStatsChunk; }

}  // namespace ditattn
