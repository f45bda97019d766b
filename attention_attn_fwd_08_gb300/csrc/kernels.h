// kernels.h -- launchers the C ABI layer (api.cu) dispatches to.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace attn {

// dt: 0 = fp32, 1 = fp16, 2 = bf16 (the attn_dtype values).
cudaError_t launch_simt_fwd(const Params& p, int dt, cudaStream_t s);
// phases: bit 1 = D = rowsum(dO*O), bit 2 = dK/dV, bit 4 = dQ
cudaError_t launch_simt_bwd(const Params& p, int dt, int phases, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const Params& p, int dt, cudaStream_t s);

// tcgen05 prefill forward / backward (fp16 / bf16; hd 64 or 128, and 32 / 96 through
// 4-D maps padded to 64 / 128).  The tensor maps are built by the caller.
struct FwdMaps {
    CUtensorMap q, k, v;
    CUtensorMap o;  // 32-row boxes, for the epilogue's stores
};
cudaError_t launch_tc_fwd_bf16(const Params& p, const FwdMaps& maps, cudaStream_t s);  // fwd_tc_bf16.cu
cudaError_t launch_tc_fwd_f16(const Params& p, const FwdMaps& maps, cudaStream_t s);   // fwd_tc_f16.cu
inline cudaError_t launch_tc_fwd(const Params& p, int dt, const FwdMaps& maps, cudaStream_t s) {
    return dt == 2 ? launch_tc_fwd_bf16(p, maps, s) : launch_tc_fwd_f16(p, maps, s);
}
struct BwdMaps {
    CUtensorMap q, dout, k, v;          // 128-row boxes
    CUtensorMap q64, dout64, k64, v64;  // 64-row boxes
    CUtensorMap o;                      // 128-row boxes (D = rowsum(dO*O) in the dQ pass)
    CUtensorMap dq32, dk32, dv32;       // 32-row boxes, for the epilogues' stores
};
cudaError_t launch_tc_bwd_bf16(const Params& p, const BwdMaps& maps, int phases, cudaStream_t s);  // bwd_tc_bf16.cu
cudaError_t launch_tc_bwd_f16(const Params& p, const BwdMaps& maps, int phases, cudaStream_t s);   // bwd_tc_f16.cu
inline cudaError_t launch_tc_bwd(const Params& p, int dt, const BwdMaps& maps, int phases, cudaStream_t s) {
    return dt == 2 ? launch_tc_bwd_bf16(p, maps, phases, s) : launch_tc_bwd_f16(p, maps, phases, s);
}

// split-KV decode (fp16 / bf16, hd 64 or 128).
struct DecMaps {
    CUtensorMap k, v;
};
cudaError_t launch_decode(const Params& p, int dt, const DecMaps& maps, cudaStream_t s);

// Fixed scratch for attn_decode_noalloc (split partials), defined in decode.cu.
constexpr size_t kDecodeScratchBytes = size_t(32) << 20;
// Device address of that scratch on the current device (looked up once per device).
cudaError_t decode_noalloc_scratch(float** out);

cudaError_t launch_selftest_wait(unsigned int* status, unsigned int timeout_us, cudaStream_t s);

// rotate-half rotary embedding of src [B][T][H*hd] into dst (src == dst: in place), hd 8 .. 256
// a multiple of 4; inverse turns every pair the other way
cudaError_t launch_rope(const void* src, void* dst, int dt, int B, int T, int H, int hd, int pos, double theta,
                        bool inverse, cudaStream_t s);
// cosine/sine table of rotary positions pos .. pos+npos-1 for the forward's fused rotation
cudaError_t launch_rope_table(float* tab, int npos, int hd, int pos, double theta, cudaStream_t s);

}  // namespace attn
