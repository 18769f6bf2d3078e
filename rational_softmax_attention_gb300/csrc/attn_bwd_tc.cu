// bf16 ra_attention backward on the tensor cores (being written).
#include "kernels.cuh"

namespace raattn {

cudaError_t launch_attn_bwd_tc(const AttnShape&, const BwdTcArgs&, const LaunchCtx&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace raattn
