// Instantiations of the attention kernel for NVFP4 Q/K + FP8 V: packed E2M1 Q/K codes with one E4M3
// scale per 16 channels of each token, applied inside BMM1 by the block-scaled tensor-core MMA, and
// one float32 scale per Q and K tensor folded into the softmax's logit scale; E4M3 V and P on the FP8
// path of BMM2; with and without Skip-Softmax. The recipe is the pages' "NVFP4 Q/K" ("VisualGen
// Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and FlashInfer backends").
#include "fmha_kernel.cuh"

namespace ditattn {

cudaError_t launch_fmha_nvfp4(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  return skip ? launch_one<QK_NVF4, PV_E4M3, 0, true>(tq, tk, tv, to, p, stream)
              : launch_one<QK_NVF4, PV_E4M3, 0, false>(tq, tk, tv, to, p, stream);
}

}  // namespace ditattn
