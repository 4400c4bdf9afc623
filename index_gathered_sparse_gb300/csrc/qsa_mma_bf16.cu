// BF16 instantiations of the tensor-core kernel (group <= 8: one 8-wide head
// tile; group <= 16: two).
#include "qsa_mma.cuh"

namespace qsa {

cudaError_t launch_mma_bf16(const Params& p, cudaStream_t s) {
  return p.group <= 8 ? launch_mma_nt<kBF16, 1>(p, s) : launch_mma_nt<kBF16, 2>(p, s);
}

int mma_ctas_per_sm_bf16(int group, bool tiles, bool umma) { return mma_occupancy<kBF16>(group, tiles, umma); }
int mma_max_clusters_bf16(int group, int splits, bool tiles, bool umma) {
  return mma_max_clusters<kBF16>(group, splits, tiles, umma);
}

}  // namespace qsa
