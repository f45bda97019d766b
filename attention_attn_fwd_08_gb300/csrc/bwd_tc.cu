// bwd_tc.cu -- placeholder until the tcgen05 backward lands.
#include "kernels.h"
namespace attn {
cudaError_t launch_tc_bwd(const Params&, int, const BwdMaps&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace attn
