// Instantiations of the attention kernel for QK16PV8: BF16 Q/K (BMM1 at full input precision),
// E4M3 V and P (BMM2 on the FP8 tensor path), with and without Skip-Softmax. The recipe is the
// pages' "QK16PV8 Attention Kernels in the CUTEDSL Backend" ("VisualGen Quantized Attention").
#include "fmha_kernel.cuh"

namespace ditattn {

cudaError_t launch_fmha_qk16pv8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  return skip ? launch_one<QK_BF16, PV_E4M3, 0, true>(tq, tk, tv, to, p, stream)
              : launch_one<QK_BF16, PV_E4M3, 0, false>(tq, tk, tv, to, p, stream);
}

// the QK16PV8 kernel of the timeout-path self-test (loads withheld)
cudaError_t launch_fmha_withheld_qk16pv8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                         const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  return launch_one<QK_BF16, PV_E4M3, 0, false, true>(tq, tk, tv, to, p, stream);
}

}  // namespace ditattn
