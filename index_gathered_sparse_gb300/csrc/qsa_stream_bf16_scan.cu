// BF16 instantiations of the persistent stream-K kernel with the scanned
// split over the tiles that hold keys.
#include "qsa_stream.cuh"

namespace qsa {

cudaError_t launch_stream_bf16_scan(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  return launch_stream_kind<kBF16, true>(p, sp, s);
}

}  // namespace qsa
