// Instantiations of the attention kernel for SAGE with FP8 E4M3 Q/K codes (K blocks 1, 4, 16).
#include "fmha_kernel.cuh"

namespace ditattn {

cudaError_t launch_fmha_sage_f8(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  if (p.k_block == 1)
    return skip ? launch_one<QK_E4M3, PV_E4M3, 1, true>(tq, tk, tv, to, p, stream)
                : launch_one<QK_E4M3, PV_E4M3, 1, false>(tq, tk, tv, to, p, stream);
  if (p.k_block == 4)
    return skip ? launch_one<QK_E4M3, PV_E4M3, 4, true>(tq, tk, tv, to, p, stream)
                : launch_one<QK_E4M3, PV_E4M3, 4, false>(tq, tk, tv, to, p, stream);
  if (p.k_block == 16)
    return skip ? launch_one<QK_E4M3, PV_E4M3, 16, true>(tq, tk, tv, to, p, stream)
                : launch_one<QK_E4M3, PV_E4M3, 16, false>(tq, tk, tv, to, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ditattn
