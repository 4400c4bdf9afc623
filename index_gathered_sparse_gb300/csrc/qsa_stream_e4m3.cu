// FP8 e4m3 instantiations of the persistent stream-K kernel.
#include "qsa_stream.cuh"

namespace qsa {

cudaError_t launch_stream_e4m3(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  return launch_stream_kind<kE4M3>(p, sp, s);
}

}  // namespace qsa
