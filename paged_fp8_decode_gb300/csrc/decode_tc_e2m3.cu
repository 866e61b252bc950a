// tcgen05 decode kernel instances for packed e2m3 KV (every row tile and Q mode
// the dispatch in decode_tc.cu can ask for).
#include "decode_tc_kernel.cuh"

namespace mj {

cudaError_t launch_tc_e2m3(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream) {
  return launch_packed<MJ_KV_E2M3>(mk, mv, p, stream);
}

}  // namespace mj
