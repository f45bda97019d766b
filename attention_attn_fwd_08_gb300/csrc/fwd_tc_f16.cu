// fwd_tc_f16.cu -- the tensor-core forwards (fwd_tc.cuh, fwd_hd256.cuh) instantiated for f16.
#include "fwd_hd256.cuh"
#include "fwd_tc.cuh"

namespace attn {

cudaError_t launch_tc_fwd_f16(const Params& p, const FwdMaps& maps, cudaStream_t s) {
    if (p.hd == 256) return fwd_hd256_typed<false>(p, maps, s);
    if (p.hd <= 64) return fwd2_typed<false, 64>(p, maps, s);
    return fwd2_typed<false, 128>(p, maps, s);
}

}  // namespace attn
