// fwd_tc.cu -- placeholder until the tcgen05 forward lands.
#include "kernels.h"
namespace attn {
cudaError_t launch_tc_fwd(const Params&, int, const FwdMaps&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace attn
