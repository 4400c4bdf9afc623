// BF16 instantiations of the persistent stream-K kernel (split without the
// scan), and the BF16 entry that picks the split the plan names.
#include "qsa_stream.cuh"

namespace qsa {

cudaError_t launch_stream_bf16(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  return sp.scan ? launch_stream_bf16_scan(p, sp, s) : launch_stream_kind<kBF16, false>(p, sp, s);
}

}  // namespace qsa
