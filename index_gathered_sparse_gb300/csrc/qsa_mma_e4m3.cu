// FP8 e4m3 instantiations of the tensor-core kernel (group <= 8: one 8-wide
// head tile; group <= 16: two).
#include "qsa_mma.cuh"

namespace qsa {

cudaError_t launch_mma_e4m3(const Params& p, cudaStream_t s) {
  return p.group <= 8 ? launch_mma_nt<kE4M3, 1>(p, s) : launch_mma_nt<kE4M3, 2>(p, s);
}

// (the tcgen05 consumer reads BF16 only: `umma` is never set here)
int mma_ctas_per_sm_e4m3(int group, bool tiles, bool umma) { return umma ? 0 : mma_occupancy<kE4M3>(group, tiles); }
int mma_max_clusters_e4m3(int group, int splits, bool tiles, bool umma) {
  return umma ? 0 : mma_max_clusters<kE4M3>(group, splits, tiles);
}

}  // namespace qsa
