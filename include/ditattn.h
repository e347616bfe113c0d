/*
 * ditattn -- diffusion-transformer attention forward pass on GB300 (sm_103a).
 *
 * The operation is full-context, non-causal multi-head attention with head_dim 128 and GQA,
 * O = softmax(Q K^T / sqrt(128)) V, in three modes that combine:
 *
 *   DENSE  BF16 Q/K/V/O ("TRTLLM Attention" user guide, section "Dense mode").
 *   SAGE   Q and K quantized per token block (INT8 or FP8 E4M3, one scale per block per head),
 *          K-smoothed (its per-channel mean over tokens subtracted) inside the routine, V
 *          quantized per channel to FP8 E4M3, and both matrix products run on low-precision
 *          tensor cores with dequantization scales ("TRTLLM Attention" user guide, section
 *          "SAGE quantization"; "VisualGen Quantized Attention", section "SageAttention in the
 *          TRTLLM backend").
 *          With qk_dtype DIT_QK_BF16, SAGE is the QK16PV8 recipe: Q and K stay BF16 (BMM1 at full
 *          input precision) and only V is quantized to FP8 E4M3, with one tensor-wide scale or one
 *          scale per channel ("VisualGen Quantized Attention", section "QK16PV8 Attention Kernels
 *          in the CUTEDSL Backend", and the quant_attention_config table: v_block_size 0 = one
 *          tensor-wide V scale, 1 = one scale per channel).
 *          With qk_dtype DIT_QK_MXFP8, SAGE is the MXFP8 Q/K + FP8 V recipe: Q and K become E4M3
 *          codes with one E8M0 (power-of-two) scale per 32 channels of each token, applied inside
 *          BMM1 by the block-scaled tensor-core MMA, and V is FP8 as in QK16PV8 ("VisualGen
 *          Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and FlashInfer backends":
 *          fixed blocks of 32 elements, q/k block sizes 0, v_block_size 0 or 1). The scale rule is
 *          the OCP Microscaling v1.0 conversion: exponent floor(log2 amax) - 8, clamped to
 *          [-127, 127]; elements round to nearest even and saturate at 448. K is not smoothed.
 *          With qk_dtype DIT_QK_NVFP4, SAGE is the NVFP4 Q/K + FP8 V recipe (same section: blocks
 *          of 16): Q and K become FP4 E2M1 codes (two per byte) with one E4M3 scale per 16 channels
 *          of each token, applied inside BMM1 by the block-scaled tensor-core MMA, and one float32
 *          scale per Q and K tensor, S = 2688 / max |x| over the tensor (NVIDIA's two-level NVFP4
 *          format); V is FP8 as in QK16PV8. K is not smoothed.
 *   SKIP   Skip-Softmax: a 128-column KV tile's exp and P.V work is skipped for a 128-row Q
 *          tile when every valid row has exp(m_tile - m_run) < threshold, with
 *          threshold = threshold_scale_factor / Skv ("SAGE + Skip-Softmax -- API Design & Test
 *          Plan", Part 1 §4, table mapping knobs to kernel arguments).
 *
 * Conventions shared by every call:
 *   - Tensors are row-major [B, S, H, 128]; Q and O have Hq heads, K and V have Hkv heads,
 *     Hq % Hkv == 0, and query head h reads kv head h / (Hq / Hkv).
 *   - All pointers named as device pointers are device memory owned by the caller; the library
 *     allocates nothing and keeps no pointer after a call returns. Tensor pointers must be
 *     16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream). Argument errors are detected on the host before anything is launched and are
 *     returned synchronously. Launch failures return DIT_E_CUDA. A kernel that finds itself
 *     waiting far longer than any correct run could take records DIT_E_TIMEOUT in a device
 *     error word and exits; dit_attn_check_errors() reports it.
 *   - The library never switches mode, dtype or backend on its own: an unsupported request is
 *     an error ("TRTLLM Attention" user guide, section "Requirements": an incompatible selection
 *     raises instead of silently changing the backend).
 *   - Only sm_103 devices (GB300 / B300) are accepted; anything else returns DIT_E_UNSUPPORTED.
 */
#ifndef DITATTN_H_
#define DITATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dit_status {
  DIT_OK = 0,
  DIT_E_INVALID_ARG = 1, /* bad shape, mode, dtype, block size, factor, or pointer alignment */
  DIT_E_UNSUPPORTED = 2, /* no CUDA device, or the current device is not sm_103 */
  DIT_E_CUDA = 3,        /* a CUDA runtime/driver call or a kernel launch failed */
  DIT_E_TIMEOUT = 4,     /* a kernel gave up waiting (reported by dit_attn_check_errors) */
  DIT_E_WORKSPACE = 5,   /* workspace missing or smaller than the *_workspace_bytes query */
  DIT_E_BOUNDS = 6       /* a library built with device-side bounds checks (DITATTN_BOUNDS_CHECK) found
                            a computed index outside its buffer and skipped that access (reported by
                            dit_attn_check_errors); never returned by the default build */
} dit_status;

/* Mode bits (or-able): DIT_MODE_SAGE | DIT_MODE_SKIP is SAGE with Skip-Softmax.
 * DIT_MODE_V_PER_TENSOR is valid only with DIT_MODE_SAGE and DIT_QK_BF16 (QK16PV8), DIT_QK_MXFP8 or
 * DIT_QK_NVFP4: V gets one
 * tensor-wide scale, max |V| over the whole [B, Skv, Hkv, 128] tensor / 448 (v_block_size 0);
 * without it V is scaled per (batch, kv head, channel) (v_block_size 1). */
enum { DIT_MODE_DENSE = 0, DIT_MODE_SAGE = 1, DIT_MODE_SKIP = 2, DIT_MODE_V_PER_TENSOR = 4 };

/* Q/K element type. DENSE uses BF16; SAGE takes INT8 or FP8 E4M3 ("TRTLLM Attention" user guide,
 * SAGE table: dtype_qk in {int8, fp8_e4m3}), BF16 for QK16PV8, MXFP8 or NVFP4 ("VisualGen
 * Quantized Attention", quant_attention_config table: qk_dtype "mxfp8", "nvfp4"). */
enum { DIT_QK_BF16 = 0, DIT_QK_INT8 = 1, DIT_QK_FP8_E4M3 = 2, DIT_QK_MXFP8 = 3, DIT_QK_NVFP4 = 4 };

/* Rows and columns of one attention tile; skip counts are kept per 128-row Q tile. */
enum { DIT_HEAD_DIM = 128, DIT_TILE = 128 };

/* Version of this interface (2: QK16PV8, DIT_MODE_V_PER_TENSOR, sage_quantize_v, the LSE outputs,
 * sage_quantize_qkv_with_mean and dit_attn_fwd_host; 3: DIT_QK_MXFP8, mx_quantize_qk and
 * dit_attn_fwd_mxfp8; 4: DIT_QK_NVFP4, nvfp4_quantize_qk and dit_attn_fwd_nvfp4). */
int dit_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* dit_status_string(dit_status status);

/*
 * Bytes of device workspace dit_attn_fwd needs for these arguments: 0 for DENSE (with or without
 * SKIP), otherwise room for the quantized codes, their scales and the K-mean / V-absmax partials
 * (QK16PV8: the V codes, V scales and V-absmax partials only; MXFP8 and NVFP4: Q/K codes and
 * scale bytes (NVFP4 also the two tensor scales), V codes, V scales and V-absmax partials).
 * Returns 0 for arguments dit_attn_fwd would reject.
 */
size_t dit_attn_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int mode, int qk_dtype, int q_block,
                                int k_block);

/*
 * The whole forward pass: (SAGE) quantize prepass, then the fused attention kernel.
 *
 *   q          device bf16 [B, Sq, Hq, 128]
 *   k, v       device bf16 [B, Skv, Hkv, 128]
 *   out        device bf16 [B, Sq, Hq, 128], written completely
 *   mode       DIT_MODE_* bits
 *   qk_dtype   DIT_QK_BF16 without SAGE; DIT_QK_INT8, DIT_QK_FP8_E4M3, (QK16PV8) DIT_QK_BF16,
 *              DIT_QK_MXFP8 or DIT_QK_NVFP4 with SAGE
 *   q_block, k_block   SAGE with INT8/FP8: tokens per Q / K scale block, each in {1, 4, 16}
 *              ("TRTLLM Attention" user guide, SAGE table); QK16PV8, MXFP8 and NVFP4: both must be
 *              0; ignored without SAGE
 *   threshold_scale_factor   with SKIP: finite and >= 0, threshold = factor / Skv (0 never
 *              skips and gives the same output as the mode without SKIP); ignored without SKIP
 *   workspace  device scratch of at least dit_attn_workspace_bytes(...) bytes, 256-byte
 *              aligned; may be NULL when that query returns 0. Its contents on entry do not
 *              matter and are garbage afterwards.
 *   skip_counts  optional device int32 [B, Hq, ceil(Sq/128)]: number of KV tiles skipped per
 *              Q tile (written as 0 without SKIP); NULL to not report
 *
 * Sq == 0 or B == 0 is a no-op. Skv must be >= 1.
 */
dit_status dit_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv, int Sq,
                        int Skv, int mode, int qk_dtype, int q_block, int k_block, float threshold_scale_factor,
                        void* stream, void* workspace, size_t workspace_bytes, int32_t* skip_counts);

/*
 * dit_attn_fwd that also writes each query row's log-sum-exp, for combining partial results
 * across devices ("VisualGen Quantized Attention", section "Requirements and behavior": a backend
 * that produces LSE composes with Attention2D / Ring context parallelism).
 *
 *   lse   device float [B, Hq, Sq], 4-byte aligned, not NULL: ln sum_j exp(s_ij) over the row's
 *         logits s_ij as the mode computes them (softmax scale applied; SAGE: from the codes and
 *         scales of the K-smoothed K, so lower by q_i . mean / sqrt(128) than for the raw K;
 *         MXFP8 and NVFP4: from the dequantized Q and K, no smoothing; with SKIP only the KV tiles
 *         that were not skipped contribute)
 * All other arguments, results and errors are those of dit_attn_fwd.
 */
dit_status dit_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                            int Hkv, int Sq, int Skv, int mode, int qk_dtype, int q_block, int k_block,
                            float threshold_scale_factor, void* stream, void* workspace, size_t workspace_bytes,
                            int32_t* skip_counts);

/*
 * Dense BF16 attention (with or without SKIP) from and to host memory, with the transfers overlapped
 * with the attention. The pages have no counterpart; this serves callers whose Q, K, V live on the
 * host (for example a step that offloads activations), so that the copies hide behind the kernels.
 *
 * The kv heads are split into `chunks` groups, each with its query heads. Every group's Q, K and V head
 * slices are copied in on h2d_stream, its attention runs on compute_stream once they have arrived, and
 * its output slice is copied back on d2h_stream once it is done: group g+1's inputs and group g-1's
 * output move while group g computes. Only the first group's inputs and the last group's output are
 * not hidden, so with chunks >= 5 and Hkv - 8 >= chunks - 4 the groups hold 1, 2 and 4 kv heads, then
 * equal shares of the rest, and 1 kv head last; otherwise they are (nearly) equal. Those two transfers
 * are made by a copy kernel when the host buffer is page-locked memory mapped for the device (its SM
 * loads and stores reach the host link's rate for narrow head slices, the copy engines do not), and
 * by the copy engines otherwise. The result equals dit_attn_fwd's bit for bit.
 *
 *   q_host, k_host, v_host, out_host   host buffers with the layouts of dit_attn_fwd (pinned memory
 *              for the copies to be asynchronous); out_host is written completely
 *   q, k, v, out   device buffers for the full tensors (16-byte aligned), used as staging
 *   mode       DIT_MODE_DENSE or DIT_MODE_SKIP; threshold_scale_factor as for dit_attn_fwd
 *   chunks     1 .. min(Hkv, 64)
 *   compute_stream, h2d_stream, d2h_stream   cudaStream_t as void*; they may be the same stream (then
 *              nothing overlaps). Work already queued on compute_stream is finished before the copies
 *              overwrite the device buffers, and the call's completion (out_host written) is signalled
 *              on compute_stream.
 * Consecutive groups' kernels alternate between compute_stream and a stream of the library's, so one
 * kernel's last partial wave overlaps the next one's first. The first call on a device creates that
 * stream and the library's events for this entry point (a one-time set-up; make it before any stream
 * capture). Calls may come from several host threads: they share those events and that stream, so
 * each call queues its work while holding a library lock, and calls queued at the same time run one
 * after the other on the library's stream.
 */
dit_status dit_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* out_host, void* q,
                             void* k, void* v, void* out, int B, int Hq, int Hkv, int Sq, int Skv, int mode,
                             float threshold_scale_factor, int chunks, void* compute_stream, void* h2d_stream,
                             void* d2h_stream);

/* Bytes of device scratch sage_quantize_qkv needs (the K-mean / V-absmax partials). */
size_t sage_quantize_workspace_bytes(int B, int Hkv, int Skv);

/*
 * The SAGE quantize prepass alone ("VisualGen Quantized Attention", section "SageAttention in
 * the TRTLLM backend": one scale per token block per head for Q/K, per head per channel for V).
 *
 *   q, k, v    device bf16 inputs as for dit_attn_fwd
 *   qk_dtype   DIT_QK_INT8 (codes are int8, |code| <= 127, round half to even) or
 *              DIT_QK_FP8_E4M3 (codes are E4M3 bit patterns, round to nearest even, saturating)
 *   q_codes    device [B, Sq, Hq, 128], 1 byte per element
 *   k_codes    device [B, Skv, Hkv, 128], codes of K minus its per-channel mean
 *   v_codes    device [B, Skv, Hkv, 128], E4M3 bit patterns
 *   q_scale    device float [B, Hq, ceil(Sq/q_block)]   = block absmax / QMAX
 *   k_scale    device float [B, Hkv, ceil(Skv/k_block)] (of the smoothed K)
 *   v_scale    device float [B, Hkv, 128]               = channel absmax / 448
 *   k_mean     device float [B, Hkv, 128]               = mean of K over all Skv tokens
 *   workspace  device scratch of sage_quantize_workspace_bytes(B, Hkv, Skv) bytes
 * QMAX is 127 for INT8 and 448 for E4M3; a block or channel whose absmax is 0 gets scale 0 and
 * zero codes (+0). Otherwise codes are those of the IEEE float32 quotient x / scale, so an E4M3
 * code of a -0 input (or of a negative quotient that rounds to zero) is 0x80. Results are
 * bit-for-bit deterministic.
 */
dit_status sage_quantize_qkv(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Sq, int Skv,
                             int qk_dtype, int q_block, int k_block, void* q_codes, void* k_codes, void* v_codes,
                             float* q_scale, float* k_scale, float* v_scale, float* k_mean, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * sage_quantize_qkv with a given K mean instead of this K's own: the global-mean option for a K
 * split across devices (context parallelism). Every shard smoothed with the mean of the whole
 * sequence gets logits shifted by the same q_i . mean / sqrt(128), so the shards' LSEs
 * (dit_attn_fwd_quantized_lse) share the shift and their partial outputs merge exactly as
 * O = sum_s exp(lse_s - lse) O_s with lse = ln sum_s exp(lse_s).
 *
 *   k_mean     device float [B, Hkv, 128], 16-byte aligned, read only (e.g. the all-reduced
 *              sums of K over every shard divided by the total token count)
 *   workspace  device scratch of sage_quantize_v_workspace_bytes(B, Hkv, Skv) bytes
 * Everything else is as for sage_quantize_qkv (INT8 or FP8 E4M3 only), minus the k_mean output.
 */
dit_status sage_quantize_qkv_with_mean(const void* q, const void* k, const void* v, const float* k_mean, int B,
                                       int Hq, int Hkv, int Sq, int Skv, int qk_dtype, int q_block, int k_block,
                                       void* q_codes, void* k_codes, void* v_codes, float* q_scale, float* k_scale,
                                       float* v_scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * sage_quantize_qkv without a workspace argument, for callers that cannot allocate device memory
 * when they call: for example a plugin whose host framework owns the whole device memory pool and
 * gives it no allocator, or a latency-critical loop where cudaMalloc (which may synchronize the
 * device) is not allowed. The pages have no counterpart; this is a library convenience.
 *
 * Inputs, outputs and results are exactly those of sage_quantize_qkv. The scratch for the K-mean
 * and V-absmax partial sums lives in a fixed 32 MiB device array inside the library, which every
 * GPU that loads the library reserves until the process exits. It holds B * Hkv * ceil(Skv/1024)
 * chunks of 128 channels at 12 bytes per channel (each of its two parts rounded up to 256 bytes);
 * larger problems return DIT_E_WORKSPACE (e.g. B * Hkv = 40 allows Skv up to about 550,000).
 * Nothing here calls cudaMalloc, cudaFree or any allocating routine.
 *
 * The first call on each device looks up the array's device address (a one-time set-up). With
 * CUDA's lazy module loading that lookup is also what loads the library's module and so reserves
 * the 32 MiB on that device: make the first call before the host framework claims its memory
 * pool, and before any stream capture. A failed lookup (e.g. no room left to reserve the array)
 * returns DIT_E_CUDA and is tried again on the next call; it is not remembered. Arguments are
 * checked first, and a problem too large for the array returns DIT_E_WORKSPACE before any
 * pointer is looked at or anything is launched. Every call shares the one array and the kernels
 * write each scratch value before reading it, so nothing needs clearing between calls; but two
 * calls whose kernels overlap on the GPU (e.g. on different streams) race on it.
 */
dit_status sage_quantize_qkv_noalloc(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Sq,
                                     int Skv, int qk_dtype, int q_block, int k_block, void* q_codes, void* k_codes,
                                     void* v_codes, float* q_scale, float* k_scale, float* v_scale, float* k_mean,
                                     void* stream);

/* Bytes of device scratch sage_quantize_v needs (the V-absmax partials). */
size_t sage_quantize_v_workspace_bytes(int B, int Hkv, int Skv);

/*
 * The QK16PV8 prepass alone: V's scales and E4M3 codes, Q and K untouched.
 *
 *   v             device bf16 [B, Skv, Hkv, 128]
 *   v_per_tensor  1: one tensor-wide scale, max |V| over the whole tensor / 448, written to every
 *                 entry of v_scale; 0: one scale per (batch, kv head, channel) = channel absmax / 448
 *   v_codes       device [B, Skv, Hkv, 128], E4M3 bit patterns of V / scale (round to nearest
 *                 even, saturating); a zero scale gives zero codes
 *   v_scale       device float [B, Hkv, 128], 16-byte aligned
 *   workspace     device scratch of sage_quantize_v_workspace_bytes(B, Hkv, Skv) bytes, 256-byte aligned
 * The codes and scales are those the QK16PV8 path of dit_attn_fwd computes, bit for bit.
 */
dit_status sage_quantize_v(const void* v, int B, int Hkv, int Skv, int v_per_tensor, void* v_codes, float* v_scale,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace dit_attn_fwd_quantized needs (INT8 codes are widened there). */
size_t dit_attn_quantized_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int qk_dtype);

/*
 * Attention over codes and scales produced by sage_quantize_qkv (same layouts and meanings).
 * mode must include DIT_MODE_SAGE; the other arguments are as for dit_attn_fwd. For QK16PV8
 * (qk_dtype DIT_QK_BF16, q_block = k_block = 0) q_codes and k_codes are the BF16 Q and K,
 * q_scale and k_scale are unused (may be NULL), and v_codes / v_scale come from sage_quantize_v.
 * MXFP8 and NVFP4 operands go through dit_attn_fwd_mxfp8 / dit_attn_fwd_nvfp4 (those qk_dtypes
 * are rejected here).
 */
dit_status dit_attn_fwd_quantized(const void* q_codes, const void* k_codes, const void* v_codes,
                                  const float* q_scale, const float* k_scale, const float* v_scale, void* out, int B,
                                  int Hq, int Hkv, int Sq, int Skv, int mode, int qk_dtype, int q_block, int k_block,
                                  float threshold_scale_factor, void* stream, void* workspace,
                                  size_t workspace_bytes, int32_t* skip_counts);

/* dit_attn_fwd_quantized that also writes each query row's LSE, as dit_attn_fwd_lse does. */
dit_status dit_attn_fwd_quantized_lse(const void* q_codes, const void* k_codes, const void* v_codes,
                                      const float* q_scale, const float* k_scale, const float* v_scale, void* out,
                                      float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int mode, int qk_dtype,
                                      int q_block, int k_block, float threshold_scale_factor, void* stream,
                                      void* workspace, size_t workspace_bytes, int32_t* skip_counts);

/*
 * The MXFP8 Q/K prepass alone ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the
 * CUTEDSL and FlashInfer backends": Q/K in fixed blocks of 32 elements along the head dimension);
 * V goes through sage_quantize_v. For every token and head, each block of 32 channels
 * 32c .. 32c+31 gets the exponent e = floor(log2 amax) - 8 of the OCP Microscaling v1.0
 * conversion (amax = the block's max |x|; e clamped to [-127, 127]; a zero block gets -127) and
 * its elements become E4M3(x / 2^e), round to nearest even, saturating at +-448.
 *
 *   q, k       device bf16 [B, Sq, Hq, 128] / [B, Skv, Hkv, 128]; q may be NULL when Sq == 0
 *   q_codes    device [B, Sq, Hq, 128] E4M3 bit patterns (16-byte aligned)
 *   k_codes    device [B, Skv, Hkv, 128] E4M3 bit patterns (16-byte aligned)
 *   q_sf       device uint8 [B, Hq, Sq, 4]: the E8M0 byte e + 127 of each block (4-byte aligned)
 *   k_sf       device uint8 [B, Hkv, Skv, 4]
 * The codes and scale bytes are those the MXFP8 path of dit_attn_fwd computes, bit for bit.
 */
dit_status mx_quantize_qk(const void* q, const void* k, int B, int Hq, int Hkv, int Sq, int Skv, void* q_codes,
                          void* k_codes, uint8_t* q_sf, uint8_t* k_sf, void* stream);

/*
 * Attention over MXFP8 Q/K (from mx_quantize_qk) and FP8 V (from sage_quantize_v, per channel or
 * tensor-wide): BMM1 applies the E8M0 block scales inside the block-scaled MMA, the rest is the
 * QK16PV8 path.
 *
 *   q_codes, k_codes, q_sf, k_sf   as mx_quantize_qk writes them
 *   v_codes, v_scale               as sage_quantize_v writes them
 *   out        device bf16 [B, Sq, Hq, 128]
 *   lse        NULL, or device float [B, Hq, Sq] (4-byte aligned) for each row's log-sum-exp, as
 *              dit_attn_fwd_lse describes
 *   mode       must include DIT_MODE_SAGE; DIT_MODE_SKIP and threshold_scale_factor as for
 *              dit_attn_fwd; DIT_MODE_V_PER_TENSOR is accepted and changes nothing here (the V
 *              scales are given)
 *   skip_counts   as for dit_attn_fwd
 * Needs no workspace. Sq == 0 or B == 0 is a no-op.
 */
dit_status dit_attn_fwd_mxfp8(const void* q_codes, const void* k_codes, const void* v_codes, const uint8_t* q_sf,
                              const uint8_t* k_sf, const float* v_scale, void* out, float* lse, int B, int Hq,
                              int Hkv, int Sq, int Skv, int mode, float threshold_scale_factor, void* stream,
                              int32_t* skip_counts);

/*
 * The NVFP4 Q/K prepass alone ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the
 * CUTEDSL and FlashInfer backends": Q/K in fixed blocks of 16 elements); V goes through
 * sage_quantize_v. Per tensor, S = 2688 / amax_T (amax_T = max |x| over the whole Q, resp. K
 * tensor; 1 if it is 0), a float32 division. Per token, head and block of 16 channels 16c..16c+15:
 * scale byte = E4M3(float32(amax_b / 6) * S) (round to nearest even, saturating), and elements
 * E2M1(float32(x * float32(S / d_b))) with d_b the byte's value (round to nearest even, saturating
 * at 6; zero codes when d_b = 0). Dequantized: x ~ code * d_b / S.
 *
 *   q, k       device bf16 [B, Sq, Hq, 128] / [B, Skv, Hkv, 128]; q may be NULL when Sq == 0
 *   q_codes    device [B, Sq, Hq, 64]: E2M1 codes, channel 2i in bits 0-3 and 2i+1 in bits 4-7 of
 *              byte i (16-byte aligned)
 *   k_codes    device [B, Skv, Hkv, 64], likewise
 *   q_sf       device uint8 [B, Hq, Sq, 8]: E4M3 block-scale bytes (8-byte aligned)
 *   k_sf       device uint8 [B, Hkv, Skv, 8]
 *   q_scale, k_scale   device float, one each: the tensor scales S (used as scratch during the call)
 * The codes, bytes and scales are those the NVFP4 path of dit_attn_fwd computes, bit for bit.
 */
dit_status nvfp4_quantize_qk(const void* q, const void* k, int B, int Hq, int Hkv, int Sq, int Skv, void* q_codes,
                             void* k_codes, uint8_t* q_sf, uint8_t* k_sf, float* q_scale, float* k_scale,
                             void* stream);

/*
 * Attention over NVFP4 Q/K (from nvfp4_quantize_qk) and FP8 V (from sage_quantize_v): BMM1 applies
 * the E4M3 block scales inside the block-scaled MMA and divides by q_scale * k_scale; the rest is the
 * QK16PV8 path. Other arguments, results and errors as for dit_attn_fwd_mxfp8.
 */
dit_status dit_attn_fwd_nvfp4(const void* q_codes, const void* k_codes, const void* v_codes, const uint8_t* q_sf,
                              const uint8_t* k_sf, const float* q_scale, const float* k_scale, const float* v_scale,
                              void* out, float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int mode,
                              float threshold_scale_factor, void* stream, int32_t* skip_counts);

/*
 * Self-test of the timeout path: launches the attention kernel (dense, or with e4m3_v = 1 the
 * QK16PV8 kernel, whose V is E4M3 codes with scales v_scale [B, Hkv, 128]) with every wait bounded by
 * wait_budget_ns and with its loads withheld: no copy into the kernel is ever issued, so the first
 * waits of the other roles run out, the kernel records DIT_E_TIMEOUT, every role leaves its loop and
 * the kernel exits with nothing in flight. `out` is not written. Returns DIT_OK once launched; the
 * following dit_attn_check_errors reports DIT_E_TIMEOUT (and clears it), and the device stays usable.
 *
 *   q, k, v, out   device buffers with the layouts of dit_attn_fwd (v: 1 byte per element if e4m3_v)
 *   wait_budget_ns 1 ms .. 10 s
 * B and Sq must be > 0.
 */
dit_status dit_selftest_withheld_loads(const void* q, const void* k, const void* v, const float* v_scale, void* out,
                                      int B, int Hq, int Hkv, int Sq, int Skv, int e4m3_v,
                                      unsigned long long wait_budget_ns, void* stream);

/*
 * Synchronizes `stream`, then reports and clears the device error word: DIT_OK, or
 * DIT_E_TIMEOUT if a kernel since the last check gave up waiting, or DIT_E_CUDA if the
 * synchronization itself failed.
 */
dit_status dit_attn_check_errors(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DITATTN_H_ */
