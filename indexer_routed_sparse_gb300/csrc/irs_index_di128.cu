// Instantiations of the persistent block-score kernel for Di = 128 (irs_index_score.cuh).
#include "irs_index_score.cuh"

namespace irs {

cudaError_t launch_score_128(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                             const CUtensorMap& tk, const IndexArgs& ia) {
  return launch_score_di<128, false>(Hi, grid, smem, st, tq, tk, ia);
}

cudaError_t configure_score_128(size_t smem) { return score_attr_all<128, false>(smem); }

}  // namespace irs
