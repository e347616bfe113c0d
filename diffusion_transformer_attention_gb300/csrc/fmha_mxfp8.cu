// Instantiations of the attention kernel for MXFP8 Q/K + FP8 V: E4M3 Q/K codes with one E8M0
// scale per 32 channels of each token, applied inside BMM1 by the block-scaled tensor-core MMA;
// E4M3 V and P on the FP8 path of BMM2; with and without Skip-Softmax. The recipe is the pages'
// "MXFP8 Q/K" ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and
// FlashInfer backends").
#include "fmha_kernel.cuh"

namespace ditattn {

cudaError_t launch_fmha_mxfp8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  return skip ? launch_one<QK_MXF8, PV_E4M3, 0, true>(tq, tk, tv, to, p, stream)
              : launch_one<QK_MXF8, PV_E4M3, 0, false>(tq, tk, tv, to, p, stream);
}

}  // namespace ditattn
