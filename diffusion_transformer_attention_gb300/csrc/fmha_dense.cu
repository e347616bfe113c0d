// Instantiations of the attention kernel for dense BF16 (with and without Skip-Softmax), and the
// dense kernel of the timeout-path self-test (loads withheld).
#include "fmha_kernel.cuh"

namespace ditattn {

cudaError_t launch_fmha_dense(bool skip, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  return skip ? launch_one<QK_BF16, PV_BF16, 0, true>(tq, tk, tv, to, p, stream)
              : launch_one<QK_BF16, PV_BF16, 0, false>(tq, tk, tv, to, p, stream);
}

cudaError_t launch_fmha_withheld_dense(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const CUtensorMap& to, const FmhaParams& p, cudaStream_t stream) {
  return launch_one<QK_BF16, PV_BF16, 0, false, true>(tq, tk, tv, to, p, stream);
}

}  // namespace ditattn
