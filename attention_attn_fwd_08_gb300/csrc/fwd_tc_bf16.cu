// fwd_tc_bf16.cu -- the tensor-core forwards (fwd_tc.cuh, fwd_hd256.cuh) instantiated for bf16.
#include "fwd_hd256.cuh"
#include "fwd_tc.cuh"

namespace attn {

cudaError_t launch_tc_fwd_bf16(const Params& p, const FwdMaps& maps, cudaStream_t s) {
    if (p.hd == 256) return fwd_hd256_typed<true>(p, maps, s);
    if (p.hd <= 64) return fwd2_typed<true, 64>(p, maps, s);
    return fwd2_typed<true, 128>(p, maps, s);
}

}  // namespace attn
