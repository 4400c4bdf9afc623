// FP8 e4m3 instantiations of the persistent stream-K kernel (split without
// the scan), and the FP8 entry that picks the split the plan names.
#include "qsa_stream.cuh"

namespace qsa {

cudaError_t launch_stream_e4m3(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  return sp.scan ? launch_stream_e4m3_scan(p, sp, s) : launch_stream_kind<kE4M3, false>(p, sp, s);
}

}  // namespace qsa
