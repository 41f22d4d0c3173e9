// Instantiations of the persistent block-score kernel for Di = 64 (irs_index_score.cuh).
#include "irs_index_score.cuh"

namespace irs {

cudaError_t launch_score_64(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                             const CUtensorMap& tk, const IndexArgs& ia) {
  return launch_score_di<64, false>(Hi, grid, smem, st, tq, tk, ia);
}

cudaError_t configure_score_64(size_t smem) { return score_attr_all<64, false>(smem); }

}  // namespace irs
