// BF16 instantiations of the persistent stream-K kernel.
#include "qsa_stream.cuh"

namespace qsa {

cudaError_t launch_stream_bf16(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  return launch_stream_kind<kBF16>(p, sp, s);
}

}  // namespace qsa
