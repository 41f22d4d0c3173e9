// Instantiations of the persistent block-score kernel with E4M3 operands, Di = 128
// (irs_index_score.cuh; Step-5 sparse page, `indexer_score_tile`: queries and summaries
// rounded to FP8 E4M3).
#include "irs_index_score.cuh"

namespace irs {

cudaError_t launch_score_e4m3(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                              const CUtensorMap& tk, const IndexArgs& ia) {
  return launch_score_di<128, true>(Hi, grid, smem, st, tq, tk, ia);
}

cudaError_t configure_score_e4m3(size_t smem) { return score_attr_all<128, true>(smem); }

}  // namespace irs
