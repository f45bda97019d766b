// bwd_tc_bf16.cu -- the tensor-core backwards (bwd_tc.cuh, bwd_hd256.cuh) instantiated for bf16.
#include "bwd_hd256.cuh"
#include "bwd_tc.cuh"

namespace attn {

cudaError_t launch_tc_bwd_bf16(const Params& p, const BwdMaps& maps, int phases, cudaStream_t s) {
    if (p.hd == 256) return bwd_hd256_typed<true>(p, maps, phases, s);
    if (p.hd <= 64) return bwd_typed<true, 64>(p, maps, phases, s);
    return bwd_typed<true, 128>(p, maps, phases, s);
}

}  // namespace attn
