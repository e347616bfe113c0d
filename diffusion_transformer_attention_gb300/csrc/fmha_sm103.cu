// Attention-kernel dispatch: picks the instantiation for the operand formats, the K scale block
// size and Skip-Softmax. The instantiations live in fmha_dense.cu, fmha_sage_i8.cu, fmha_sage_f8.cu
// fmha_qk16pv8.cu, fmha_mxfp8.cu and fmha_nvfp4.cu so that they compile in parallel.
#include "ditattn_internal.h"

namespace ditattn {

cudaError_t launch_fmha(int qk_format, int pv_format, bool skip, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  if (qk_format == QK_BF16 && pv_format == PV_BF16) return launch_fmha_dense(skip, tq, tk, tv, to, p, stream);
  if (qk_format == QK_F16 && pv_format == PV_E4M3) return launch_fmha_sage_i8(skip, tq, tk, tv, to, p, stream);
  if (qk_format == QK_E4M3 && pv_format == PV_E4M3) return launch_fmha_sage_f8(skip, tq, tk, tv, to, p, stream);
  if (qk_format == QK_BF16 && pv_format == PV_E4M3) return launch_fmha_qk16pv8(skip, tq, tk, tv, to, p, stream);
  if (qk_format == QK_MXF8 && pv_format == PV_E4M3) return launch_fmha_mxfp8(skip, tq, tk, tv, to, p, stream);
  if (qk_format == QK_NVF4 && pv_format == PV_E4M3) return launch_fmha_nvfp4(skip, tq, tk, tv, to, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fmha_withheld(int pv_format, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  if (pv_format == PV_BF16) return launch_fmha_withheld_dense(tq, tk, tv, to, p, stream);
  if (pv_format == PV_E4M3) return launch_fmha_withheld_qk16pv8(tq, tk, tv, to, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ditattn
