// tcgen05 decode kernel instances for e4m3 KV, head size 128 (every row tile and Q mode
// the dispatch in decode_tc.cu can ask for).
#include "decode_tc_kernel.cuh"

namespace mj {

cudaError_t launch_tc_e4m3_d128(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream) {
  if (p.q_mode == MJ_Q_BF16) return launch_rows<MJ_KV_E4M3, 1>(mk, mv, p, stream);
  if (p.q_mode == MJ_Q_FP8_FUSED) return launch_rows<MJ_KV_E4M3, 2>(mk, mv, p, stream);
  return launch_rows<MJ_KV_E4M3, 0>(mk, mv, p, stream);
}

}  // namespace mj
