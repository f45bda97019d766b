// api.cu -- the C ABI declared in include/attn.h: host-side validation,
// planning (tile and split counts), TMA descriptor encoding and dispatch.
//
// Argument rules follow ferrotensor engine/attention.rs, AttentionDims::new
// (num_heads a multiple of num_kv_heads, bounded head_dim) and the brotensor
// ops/flash_attention.h contracts (caller-owned buffers, overwrite semantics,
// a length-Tk fp32 key mask).  Nothing here allocates, frees or synchronises
// (except attn_get_device_status, which exists to read the status word).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"

using namespace attn;


namespace {

constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_launches{0};

attn_status counted(cudaError_t e, int kernels) {
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add((unsigned long long)kernels, std::memory_order_relaxed);
    return ATTN_OK;
}

// Device status word: bounded waits that run out OR a bit in here.
__device__ unsigned int g_status_word;

unsigned int* status_ptr() {
    static unsigned int* ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned int*>(p);
    }
    return ptrs[dev];
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D map over a [batches][rows][inner] 16-bit tensor, box {64, box_rows, 1},
// 128-byte swizzle (inner box = 64 elements = 128 bytes).  Rows lie row_stride
// elements apart (inner when 0): a map over some columns of wider rows.
bool make_map(CUtensorMap* m, int dt, const void* base, long long inner, long long rows, long long batches,
              int box_rows, long long row_stride = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const CUtensorMapDataType t = dt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const long long rs = row_stride > 0 ? row_stride : inner;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)batches};
    cuuint64_t strides[2] = {(cuuint64_t)rs * 2, (cuuint64_t)rs * rows * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, t, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over a [batches][rows][heads][hd] 16-bit tensor, box {64, 1, box_rows, 1},
// 128-byte swizzle: for a head size below the kernel's (32 in a 64 kernel, 96 in a
// 128 kernel), the box's columns past hd load as zeros and are never stored.
bool make_map4(CUtensorMap* m, int dt, const void* base, int hd, long long heads, long long rows,
               long long batches, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const CUtensorMapDataType t = dt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)heads, (cuuint64_t)rows, (cuuint64_t)batches};
    cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)heads * hd * 2, (cuuint64_t)rows * heads * hd * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, t, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------- validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// decode_hd: a decode entry point, whose 16-bit split kernel is built for hd 64, 128, 256
attn_status check_common(attn_dtype dt, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale, int causal,
                         int window, float softcap, int q_offset, const float* key_mask, long long mstride,
                         bool decode_hd = false) {
    if (dt != ATTN_F32 && dt != ATTN_F16 && dt != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (B < 0 || Tq < 0 || Tk < 0) return ATTN_ERR_INVALID_ARG;
    if (B > 65535) return ATTN_ERR_INVALID_ARG;
    if (H <= 0 || Hkv <= 0 || H % Hkv != 0 || H > 65535) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !isfinite(softcap)) return ATTN_ERR_INVALID_ARG;
    if (window < 0 || q_offset < 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (mstride < 0) return ATTN_ERR_INVALID_ARG;
    if (key_mask && (reinterpret_cast<uintptr_t>(key_mask) & 3u)) return ATTN_ERR_INVALID_ARG;
    if ((long long)Tq + q_offset > INT32_MAX - 1) return ATTN_ERR_INVALID_ARG;
    // head sizes: 32, 64, 96, 128 and 256 (16-bit on the tensor cores, fp32 on the
    // CUDA-core kernels); the 16-bit decode split kernel takes 64, 128 and 256
    if (hd != 32 && hd != 64 && hd != 96 && hd != 128 && hd != 256) return ATTN_ERR_UNSUPPORTED;
    if (decode_hd && dt != ATTN_F32 && hd != 64 && hd != 128 && hd != 256) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

Params base_params(int B, int Tq, int Tk, int H, int Hkv, int hd, float scale, int causal, int window,
                   float softcap, int q_offset, const float* key_mask, long long mstride) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.B = B; p.Tq = Tq; p.Tk = Tk; p.H = H; p.Hkv = Hkv; p.hd = hd; p.G = H / Hkv;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    // causal, window (ferrotensor's |p - j| < window) as the two-sided window
    p.wl = window > 0 ? window - 1 : -1;
    p.wr = causal ? 0 : (window > 0 ? window - 1 : -1);
    p.softcap = softcap; p.q_offset = q_offset;
    p.key_mask = key_mask; p.mask_bstride = mstride;
    p.status = status_ptr();
    return p;
}

// fp16/bf16 at hd 64 / 128 run on the tensor cores, and so do hd 32 and 96 as 64 and
// 128 with the columns past the head read as zeros (dense batches; packed sequences
// and a score bias at those sizes take the CUDA-core kernels).  fp32 stays on the
// CUDA-core kernels (no TF32, no 16-bit P), which is what fp32 accuracy needs.
bool padded_head(int hd) { return hd == 32 || hd == 96; }
bool use_tcgen05(attn_dtype dt, int hd) { return dt != ATTN_F32 && (hd == 32 || hd == 64 || hd == 96 || hd == 128); }

// 16-bit hd 256 also runs on the tensor cores in dense batches without a bias (the
// forward one query tile per work item; the backward in separate dV, dK and dQ passes).
bool use_tc_fwd(attn_dtype dt, int hd) { return use_tcgen05(dt, hd) || (dt != ATTN_F32 && hd == 256); }

// Tensor map of one activation for the tensor-core kernels: 3-D at hd 64 / 128, 4-D
// (zero-filled past the head) at hd 32 / 96.  A row stride (elements; 0 = heads*hd)
// maps the activation's columns inside wider rows (3-D maps only).
bool act_map(CUtensorMap* m, attn_dtype dt, const void* base, int hd, long long heads, long long rows,
             long long batches, int box_rows, long long row_stride = 0) {
    if (padded_head(hd)) return row_stride == 0 && make_map4(m, (int)dt, base, hd, heads, rows, batches, box_rows);
    return make_map(m, (int)dt, base, heads * hd, rows, batches, box_rows, row_stride);
}

// Decode split plan: a deterministic function of the shape.  Aim for about
// eight waves of two resident CTAs on each of GB300's 152 SMs.
void decode_plan(int B, int Lq, int Tk, int H, int Hkv, int* splits, int* chunk) {
    const int R = (H / Hkv) * Lq;
    const long long units = (long long)B * Hkv * ((R + 15) / 16);
    const long long target = 8LL * 2 * 152;
    long long s = (target + units - 1) / units;
    const long long max_s = Tk > 0 ? (Tk + 63) / 64 : 1;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    long long c = Tk > 0 ? (Tk + s - 1) / s : 64;
    c = ((c + 63) / 64) * 64;
    *chunk = (int)c;
    *splits = Tk > 0 ? (int)((Tk + c - 1) / c) : 1;
}

// O = 0, LSE = -inf for every row (Tk == 0: no key is visible).
template <typename T>
__global__ void fill_empty_kernel(T* o, long long n_o, float* lse, long long n_lse) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i < n_o) o[i] = T(0.f);
    if (lse && i < n_lse) lse[i] = -INFINITY;
}

attn_status fill_empty(attn_dtype dt, void* o, long long n_o, float* lse, long long n_lse, cudaStream_t s) {
    const long long n = n_o > n_lse ? n_o : n_lse;
    if (n == 0) return ATTN_OK;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    if (dt == ATTN_F32) fill_empty_kernel<float><<<blocks, 256, 0, s>>>((float*)o, n_o, lse, n_lse);
    else if (dt == ATTN_F16) fill_empty_kernel<__half><<<blocks, 256, 0, s>>>((__half*)o, n_o, lse, n_lse);
    else fill_empty_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>((__nv_bfloat16*)o, n_o, lse, n_lse);
    return counted(cudaGetLastError(), 1);
}

size_t elem_size(attn_dtype dt) { return dt == ATTN_F32 ? 4 : 2; }

}  // namespace

// ================================================================ C ABI
extern "C" {

int attn_abi_version(void) { return 1; }

const char* attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    }
    return "unknown status";
}

int attn_kernel_family(attn_dtype dt, int hd) { return use_tc_fwd(dt, hd) ? 1 : 0; }

int attn_kernel_family_bwd(attn_dtype dt, int hd) { return use_tc_fwd(dt, hd) ? 1 : 0; }

}  // extern "C"

namespace {

// The forward once the arguments are checked and the window set in p.  With
// in_stride > 0 the rows of q, k and v lie in_stride elements apart (the tensor-core
// kernels only: the caller routes such calls there).
attn_status fwd_launch(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse, Params p,
                       void* stream, long long in_stride = 0) {
    const int B = p.B, Tq = p.Tq, Tk = p.Tk, H = p.H, Hkv = p.Hkv, hd = p.hd;
    if (B == 0 || Tq == 0) return ATTN_OK;
    if (!q || !o || (Tk > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (Tk == 0)
        return fill_empty(dt, o, (long long)B * Tq * H * hd, lse, lse ? (long long)B * H * Tq : 0, s);
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    // a bias or packed fused-QKV rows at the padded head sizes or at hd 256 take the
    // CUDA-core kernels
    if (!use_tc_fwd(dt, hd) || ((p.bias || p.row_bounds) && (padded_head(hd) || hd == 256)))
        return counted(launch_simt_fwd(p, (int)dt, s), 1);
    FwdMaps maps;
    const int kv_rows = hd == 256 ? 64 : 128;  // keys per tile
    if (!act_map(&maps.q, dt, q, hd, H, Tq, B, 128, in_stride) ||
        !act_map(&maps.k, dt, k, hd, Hkv, Tk, B, kv_rows, in_stride) ||
        !act_map(&maps.v, dt, v, hd, Hkv, Tk, B, kv_rows, in_stride) || !act_map(&maps.o, dt, o, hd, H, Tq, B, 32))
        return ATTN_ERR_CUDA;
    return counted(launch_tc_fwd(p, (int)dt, maps, s), 1);
}

}  // namespace

extern "C" {

attn_status attn_fwd(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Tq, int Tk, int H, int Hkv, int hd, float scale, int causal, int window, float softcap,
                     int q_offset, const float* key_mask, long long key_mask_bstride, void* stream) {
    attn_status st = check_common(dt, B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride);
    if (st != ATTN_OK) return st;
    return fwd_launch(dt, q, k, v, o, lse,
                      base_params(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride),
                      stream);
}

size_t attn_bwd_workspace_size(int B, int Tq, int H) {
    if (B < 0 || Tq < 0 || H < 0) return 0;
    const size_t tq_pad = ((size_t)Tq + 63) / 64 * 64;
    return 2 * (size_t)B * H * tq_pad * sizeof(float);  // D and LSE*log2(e), rows padded to 64
}

}  // extern "C"

namespace {

// The backward once the arguments are checked and the window set in p.  With
// in_stride / grad_stride > 0 the rows of q, k, v / of dq, dk, dv lie that many
// elements apart (the tensor-core kernels only: the caller routes such calls there).
attn_status bwd_launch(attn_dtype dt, const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                       Params p, void* stream, int phases, long long in_stride = 0, long long grad_stride = 0) {
    const int B = p.B, Tq = p.Tq, Tk = p.Tk, H = p.H, Hkv = p.Hkv, hd = p.hd;
    if (phases <= 0 || phases > 7) return ATTN_ERR_INVALID_ARG;
    if (B == 0) return ATTN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(dt);
    if (Tq == 0 || Tk == 0) {
        // no visible pair: every gradient is zero
        if (Tk > 0 && (phases & 2)) {
            if (!dk || !dv || !aligned16(dk) || !aligned16(dv)) return ATTN_ERR_INVALID_ARG;
            const size_t n = (size_t)B * Tk * Hkv * hd * es;
            if (cudaMemsetAsync(dk, 0, n, s) != cudaSuccess || cudaMemsetAsync(dv, 0, n, s) != cudaSuccess)
                return ATTN_ERR_CUDA;
        }
        if (Tq > 0 && (phases & 4)) {
            if (!dq || !aligned16(dq)) return ATTN_ERR_INVALID_ARG;
            if (cudaMemsetAsync(dq, 0, (size_t)B * Tq * H * hd * es, s) != cudaSuccess) return ATTN_ERR_CUDA;
        }
        return ATTN_OK;
    }
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
    if (workspace_bytes < attn_bwd_workspace_size(B, Tq, H)) return ATTN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    for (const void* x : ptrs)
        if (!aligned16(x)) return ATTN_ERR_INVALID_ARG;
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o_in = o; p.dout = dout; p.lse_in = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    p.tq_pad = (Tq + 63) / 64 * 64;
    p.ndelta = static_cast<float*>(workspace);
    p.nlse2 = p.ndelta + (size_t)B * H * p.tq_pad;
    if (!use_tc_fwd(dt, hd) || ((p.bias || p.row_bounds) && (padded_head(hd) || hd == 256))) {
        // the fp32 dQ pass reads D from the workspace: pass 4 implies pass 1 there
        const int ph = (phases & 4) ? (phases | 1) : phases;
        const int nks = ((ph & 1) ? 1 : 0) + ((ph & 2) ? 1 : 0) + ((ph & 4) ? 1 : 0);
        return counted(launch_simt_bwd(p, (int)dt, ph, s), nks);
    }
    // the tensor-core dQ pass forms D itself: pass 1 is then not run separately (at hd
    // 256 the preprocess runs for passes 1 and 4, and dK and dV are two launches)
    const int nk = hd == 256 ? ((phases & 5) ? 1 : 0) + ((phases & 2) ? 2 : 0) + ((phases & 4) ? 1 : 0)
                             : ((phases & 1) && !(phases & 4) ? 1 : 0) + ((phases & 2) ? 1 : 0) + ((phases & 4) ? 1 : 0);
    BwdMaps maps;
    const long long is = in_stride, gs = grad_stride;
    if (!act_map(&maps.q, dt, q, hd, H, Tq, B, 128, is) || !act_map(&maps.dout, dt, dout, hd, H, Tq, B, 128) ||
        !act_map(&maps.k, dt, k, hd, Hkv, Tk, B, 128, is) || !act_map(&maps.v, dt, v, hd, Hkv, Tk, B, 128, is) ||
        !act_map(&maps.q64, dt, q, hd, H, Tq, B, 64, is) || !act_map(&maps.dout64, dt, dout, hd, H, Tq, B, 64) ||
        !act_map(&maps.k64, dt, k, hd, Hkv, Tk, B, 64, is) || !act_map(&maps.v64, dt, v, hd, Hkv, Tk, B, 64, is) ||
        ((phases & 4) &&
         (!act_map(&maps.dq32, dt, dq, hd, H, Tq, B, 32, gs) || !act_map(&maps.o, dt, o, hd, H, Tq, B, 128))) ||
        ((phases & 2) &&
         (!act_map(&maps.dk32, dt, dk, hd, Hkv, Tk, B, 32, gs) || !act_map(&maps.dv32, dt, dv, hd, Hkv, Tk, B, 32, gs))))
        return ATTN_ERR_CUDA;
    return counted(launch_tc_bwd(p, (int)dt, maps, phases, s), nk);
}

}  // namespace

extern "C" {

attn_status attn_bwd_phases(attn_dtype dt, const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale,
                            int causal, int window, float softcap, int q_offset, const float* key_mask,
                            long long key_mask_bstride, void* stream, int phases) {
    attn_status st = check_common(dt, B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride);
    if (st != ATTN_OK) return st;
    return bwd_launch(dt, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                      base_params(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride),
                      stream, phases);
}

attn_status attn_bwd(attn_dtype dt, const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                     int Tq, int Tk, int H, int Hkv, int hd, float scale, int causal, int window, float softcap,
                     int q_offset, const float* key_mask, long long key_mask_bstride, void* stream) {
    return attn_bwd_phases(dt, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Tq, Tk, H, Hkv,
                           hd, scale, causal, window, softcap, q_offset, key_mask, key_mask_bstride, stream, 7);
}

// ------------------------------------------------------ packed sequences
// The dense kernels run on the packed tensors as one batch of total rows; each
// work item reads its sequence's bounds from cu_seqlens on the device (Seq in
// common.cuh).  Launch shapes come from batch and the max_seqlen bounds.
namespace {

attn_status check_varlen(attn_dtype dt, const int* cu_q, const int* cu_k, int batch, int max_q, int max_k,
                         int total_q, int total_k, int H, int Hkv, int hd, float scale, int causal, int window,
                         float softcap) {
    attn_status st = check_common(dt, batch, max_q, max_k, H, Hkv, hd, scale, causal, window, softcap, 0, nullptr, 0);
    if (st != ATTN_OK) return st;
    if (total_q < 0 || total_k < 0 || max_q > total_q || max_k > total_k) return ATTN_ERR_INVALID_ARG;
    if (batch > 0 && (!cu_q || !cu_k)) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_k) & 3u))
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

Params varlen_params(const int* cu_q, const int* cu_k, int batch, int max_q, int max_k, int total_q, int total_k,
                     int H, int Hkv, int hd, float scale, int causal, int window, float softcap) {
    Params p = base_params(batch, max_q, max_k, H, Hkv, hd, scale, causal, window, softcap, 0, nullptr, 0);
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.total_q = total_q;
    p.total_k = total_k;
    return p;
}

}  // namespace

attn_status attn_varlen_fwd(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int max_seqlen_q,
                            int max_seqlen_k, int total_q, int total_k, int H, int Hkv, int hd, float scale,
                            int causal, int window, float softcap, void* stream) {
    attn_status st = check_varlen(dt, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k, total_q,
                                  total_k, H, Hkv, hd, scale, causal, window, softcap);
    if (st != ATTN_OK) return st;
    if (batch == 0 || max_seqlen_q == 0 || total_q == 0) return ATTN_OK;
    if (!q || !o || (total_k > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Params p = varlen_params(cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k, total_q, total_k, H,
                             Hkv, hd, scale, causal, window, softcap);
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    // no keys anywhere: the CUDA-core kernel writes O = 0 and LSE = -inf per row
    if (!use_tcgen05(dt, hd) || padded_head(hd) || max_seqlen_k == 0 || total_k == 0)
        return counted(launch_simt_fwd(p, (int)dt, s), 1);
    FwdMaps maps;
    if (!make_map(&maps.q, dt, q, (long long)H * hd, total_q, 1, 128) ||
        !make_map(&maps.k, dt, k, (long long)Hkv * hd, total_k, 1, 128) ||
        !make_map(&maps.v, dt, v, (long long)Hkv * hd, total_k, 1, 128) ||
        !make_map(&maps.o, dt, o, (long long)H * hd, total_q, 1, 32))
        return ATTN_ERR_CUDA;
    return counted(launch_tc_fwd(p, (int)dt, maps, s), 1);
}

attn_status attn_varlen_bwd(attn_dtype dt, const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                            int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int H, int Hkv, int hd,
                            float scale, int causal, int window, float softcap, void* stream) {
    attn_status st = check_varlen(dt, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k, total_q,
                                  total_k, H, Hkv, hd, scale, causal, window, softcap);
    if (st != ATTN_OK) return st;
    if (batch == 0 || (total_q == 0 && total_k == 0)) return ATTN_OK;
    const size_t ws_need = attn_bwd_workspace_size(batch, max_seqlen_q, H);
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || (!workspace && ws_need > 0))
        return ATTN_ERR_INVALID_ARG;
    if (workspace_bytes < ws_need) return ATTN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    for (const void* x : ptrs)
        if (!aligned16(x)) return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Params p = varlen_params(cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k, total_q, total_k, H,
                             Hkv, hd, scale, causal, window, softcap);
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o_in = o; p.dout = dout; p.lse_in = lse;
    p.dq = dq; p.dk = dk; p.dv = dv;
    p.tq_pad = (max_seqlen_q + 63) / 64 * 64;
    p.ndelta = static_cast<float*>(workspace);
    p.nlse2 = p.ndelta + (size_t)batch * H * p.tq_pad;
    // with no query rows or no key rows anywhere, the CUDA-core kernels write the
    // zero gradients of whatever rows the sequences have
    if (!use_tcgen05(dt, hd) || padded_head(hd) || max_seqlen_q == 0 || max_seqlen_k == 0 || total_q == 0 ||
        total_k == 0)
        return counted(launch_simt_bwd(p, (int)dt, 7, s), 3);
    BwdMaps maps;
    if (!make_map(&maps.q, dt, q, (long long)H * hd, total_q, 1, 128) ||
        !make_map(&maps.dout, dt, dout, (long long)H * hd, total_q, 1, 128) ||
        !make_map(&maps.k, dt, k, (long long)Hkv * hd, total_k, 1, 128) ||
        !make_map(&maps.v, dt, v, (long long)Hkv * hd, total_k, 1, 128) ||
        !make_map(&maps.q64, dt, q, (long long)H * hd, total_q, 1, 64) ||
        !make_map(&maps.dout64, dt, dout, (long long)H * hd, total_q, 1, 64) ||
        !make_map(&maps.k64, dt, k, (long long)Hkv * hd, total_k, 1, 64) ||
        !make_map(&maps.v64, dt, v, (long long)Hkv * hd, total_k, 1, 64) ||
        !make_map(&maps.dq32, dt, dq, (long long)H * hd, total_q, 1, 32) ||
        !make_map(&maps.o, dt, o, (long long)H * hd, total_q, 1, 128) ||
        !make_map(&maps.dk32, dt, dk, (long long)Hkv * hd, total_k, 1, 32) ||
        !make_map(&maps.dv32, dt, dv, (long long)Hkv * hd, total_k, 1, 32))
        return ATTN_ERR_CUDA;
    return counted(launch_tc_bwd(p, (int)dt, maps, 7, s), 2);
}

// ----------------------------------------- two-sided window, additive bias
}  // extern "C"

namespace {

// Params of an _ex call: the window sides (negative = unbounded) and the bias.
attn_status ex_params(attn_dtype dt, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale, int window_left,
                      int window_right, float softcap, int q_offset, const float* key_mask, long long mstride,
                      const float* bias, long long sb, long long sh, long long sq, long long sk, Params* out) {
    attn_status st = check_common(dt, B, Tq, Tk, H, Hkv, hd, scale, 0, 0, softcap, q_offset, key_mask, mstride);
    if (st != ATTN_OK) return st;
    if (bias && ((reinterpret_cast<uintptr_t>(bias) & 3u) || sb < 0 || sh < 0 || sq < 0 || sk < 0))
        return ATTN_ERR_INVALID_ARG;
    Params p = base_params(B, Tq, Tk, H, Hkv, hd, scale, 0, 0, softcap, q_offset, key_mask, mstride);
    p.wl = window_left < 0 ? -1 : window_left;
    p.wr = window_right < 0 ? -1 : window_right;
    p.bias = bias;
    p.bias_sb = sb; p.bias_sh = sh; p.bias_sq = sq; p.bias_sk = sk;
    *out = p;
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd_ex(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Tq, int Tk, int H, int Hkv, int hd, float scale, int window_left, int window_right,
                        float softcap, int q_offset, const float* key_mask, long long key_mask_bstride,
                        const float* bias, long long bias_sb, long long bias_sh, long long bias_sq,
                        long long bias_sk, void* stream) {
    Params p;
    attn_status st = ex_params(dt, B, Tq, Tk, H, Hkv, hd, scale, window_left, window_right, softcap, q_offset,
                               key_mask, key_mask_bstride, bias, bias_sb, bias_sh, bias_sq, bias_sk, &p);
    if (st != ATTN_OK) return st;
    return fwd_launch(dt, q, k, v, o, lse, p, stream);
}

attn_status attn_bwd_ex(attn_dtype dt, const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                        size_t workspace_bytes, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale,
                        int window_left, int window_right, float softcap, int q_offset, const float* key_mask,
                        long long key_mask_bstride, const float* bias, long long bias_sb, long long bias_sh,
                        long long bias_sq, long long bias_sk, void* stream) {
    Params p;
    attn_status st = ex_params(dt, B, Tq, Tk, H, Hkv, hd, scale, window_left, window_right, softcap, q_offset,
                               key_mask, key_mask_bstride, bias, bias_sb, bias_sh, bias_sq, bias_sk, &p);
    if (st != ATTN_OK) return st;
    return bwd_launch(dt, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, p, stream, 7);
}

attn_status attn_rope(attn_dtype dt, void* x, int B, int T, int H, int hd, int pos, float theta, void* stream) {
    if (dt != ATTN_F32 && dt != ATTN_F16 && dt != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || H <= 0 || H > 65535 || pos < 0 || !(theta > 0.f) || !isfinite(theta))
        return ATTN_ERR_INVALID_ARG;
    if (hd < 4 || hd > 256 || hd % 4) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || T == 0) return ATTN_OK;
    if (!x || !aligned16(x)) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * T > (long long)INT32_MAX * 8) return ATTN_ERR_UNSUPPORTED;
    return counted(
        launch_rope(x, x, (int)dt, B, T, H, hd, pos, (double)theta, false, static_cast<cudaStream_t>(stream)), 1);
}

}  // extern "C"

// --------------------------------------------------- rotary embedding fused
namespace {

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// rotary positions the table covers: query row i sits at q_offset + i, key j at j
long long rope_npos(int Tq, int Tk, int q_offset) {
    const long long a = (long long)q_offset + Tq;
    return a > Tk ? a : Tk;
}

// the forward turns the query tiles inside the kernel (16-bit, hd 64 / 128); other
// types and head sizes turn q into the workspace first
bool rope_in_kernel(attn_dtype dt, int hd) { return dt != ATTN_F32 && (hd == 64 || hd == 128); }

bool rope_args_ok(attn_dtype dt, int hd, int rope_pos, float theta) {
    if (rope_pos < 0 || !(theta > 0.f) || !isfinite(theta)) return false;
    (void)dt;
    return hd % 4 == 0 && hd >= 4 && hd <= 256;
}

}  // namespace

extern "C" {

size_t attn_fwd_rope_workspace_size(attn_dtype dt, int B, int Tq, int Tk, int H, int Hkv, int hd, int q_offset) {
    if (B < 0 || Tq < 0 || Tk < 0 || H <= 0 || Hkv <= 0 || hd <= 0 || q_offset < 0) return 0;
    const size_t es = elem_size(dt);
    size_t n = align256((size_t)B * Tk * Hkv * hd * es);  // rotated k
    if (rope_in_kernel(dt, hd)) n += align256((size_t)rope_npos(Tq, Tk, q_offset) * hd * sizeof(float));
    else n += align256((size_t)B * Tq * H * hd * es);  // rotated q
    return n;
}

attn_status attn_fwd_rope(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                          void* workspace, size_t workspace_bytes, int B, int Tq, int Tk, int H, int Hkv, int hd,
                          float scale, int causal, int window, float softcap, int q_offset, const float* key_mask,
                          long long key_mask_bstride, int rope_pos, float rope_theta, void* stream) {
    attn_status st = check_common(dt, B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride);
    if (st != ATTN_OK) return st;
    if (!rope_args_ok(dt, hd, rope_pos, rope_theta)) return ATTN_ERR_INVALID_ARG;
    if ((long long)rope_pos + rope_npos(Tq, Tk, q_offset) > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    if (B == 0 || Tq == 0) return ATTN_OK;
    Params p = base_params(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                           key_mask_bstride);
    if (Tk == 0) return fwd_launch(dt, q, k, v, o, lse, p, stream);
    if (!workspace || !aligned16(workspace) || !k || !q ||
        workspace_bytes < attn_fwd_rope_workspace_size(dt, B, Tq, Tk, H, Hkv, hd, q_offset))
        return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k)) return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(dt);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* k_rot = ws;
    uint8_t* rest = ws + align256((size_t)B * Tk * Hkv * hd * es);
    // keys at rotary positions rope_pos + j
    if (launch_rope(k, k_rot, (int)dt, B, Tk, Hkv, hd, rope_pos, (double)rope_theta, false, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (rope_in_kernel(dt, hd)) {
        float* tab = reinterpret_cast<float*>(rest);
        const int npos = (int)rope_npos(Tq, Tk, q_offset);
        if (launch_rope_table(tab, npos, hd, rope_pos, (double)rope_theta, s) != cudaSuccess) return ATTN_ERR_CUDA;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        p.rope_tab = tab;
        p.rope_npos = npos;
        return fwd_launch(dt, q, k_rot, v, o, lse, p, stream);
    }
    // queries at rotary positions rope_pos + q_offset + i, turned into the workspace
    void* q_rot = rest;
    if (launch_rope(q, q_rot, (int)dt, B, Tq, H, hd, rope_pos + q_offset, (double)rope_theta, false, s) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return fwd_launch(dt, q_rot, k_rot, v, o, lse, p, stream);
}

size_t attn_bwd_rope_workspace_size(attn_dtype dt, int B, int Tq, int Tk, int H, int Hkv, int hd) {
    if (B < 0 || Tq < 0 || Tk < 0 || H <= 0 || Hkv <= 0 || hd <= 0) return 0;
    const size_t es = elem_size(dt);
    return align256((size_t)B * Tq * H * hd * es) + align256((size_t)B * Tk * Hkv * hd * es) +
           align256(attn_bwd_workspace_size(B, Tq, H));
}

attn_status attn_bwd_rope(attn_dtype dt, const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                          size_t workspace_bytes, int B, int Tq, int Tk, int H, int Hkv, int hd, float scale,
                          int causal, int window, float softcap, int q_offset, const float* key_mask,
                          long long key_mask_bstride, int rope_pos, float rope_theta, void* stream) {
    attn_status st = check_common(dt, B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride);
    if (st != ATTN_OK) return st;
    if (!rope_args_ok(dt, hd, rope_pos, rope_theta)) return ATTN_ERR_INVALID_ARG;
    if ((long long)rope_pos + rope_npos(Tq, Tk, q_offset) > INT32_MAX) return ATTN_ERR_INVALID_ARG;
    if (B == 0) return ATTN_OK;
    Params p = base_params(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                           key_mask_bstride);
    if (Tq == 0 || Tk == 0)  // no visible pair: zero gradients, nothing to turn
        return bwd_launch(dt, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, p, stream, 7);
    if (!workspace || !aligned16(workspace) || !q || !k || !dq || !dk ||
        workspace_bytes < attn_bwd_rope_workspace_size(dt, B, Tq, Tk, H, Hkv, hd))
        return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(dq) || !aligned16(dk)) return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(dt);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* q_rot = ws;
    void* k_rot = ws + align256((size_t)B * Tq * H * hd * es);
    void* ws_bwd = static_cast<uint8_t*>(k_rot) + align256((size_t)B * Tk * Hkv * hd * es);
    // the forward's rotated operands, the backward on them, then the gradients turned
    // back (dL/dq = R^T dL/d(Rq): the inverse turn at the same positions)
    if (launch_rope(q, q_rot, (int)dt, B, Tq, H, hd, rope_pos + q_offset, (double)rope_theta, false, s) !=
            cudaSuccess ||
        launch_rope(k, k_rot, (int)dt, B, Tk, Hkv, hd, rope_pos, (double)rope_theta, false, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    g_launches.fetch_add(2, std::memory_order_relaxed);
    st = bwd_launch(dt, q_rot, k_rot, v, o, dout, lse, dq, dk, dv, ws_bwd, attn_bwd_workspace_size(B, Tq, H), p,
                    stream, 7);
    if (st != ATTN_OK) return st;
    if (launch_rope(dq, dq, (int)dt, B, Tq, H, hd, rope_pos + q_offset, (double)rope_theta, true, s) != cudaSuccess ||
        launch_rope(dk, dk, (int)dt, B, Tk, Hkv, hd, rope_pos, (double)rope_theta, true, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    g_launches.fetch_add(2, std::memory_order_relaxed);
    return ATTN_OK;
}

unsigned long long attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

attn_status attn_decode_plan(int B, int Lq, int Tk, int H, int Hkv, int* splits, int* chunk) {
    if (!splits || !chunk || B <= 0 || Lq <= 0 || Tk < 0 || H <= 0 || Hkv <= 0 || H % Hkv) return ATTN_ERR_INVALID_ARG;
    decode_plan(B, Lq, Tk, H, Hkv, splits, chunk);
    return ATTN_OK;
}

size_t attn_decode_workspace_size(int B, int Lq, int Tk, int H, int Hkv, int hd) {
    if (B <= 0 || Lq <= 0 || Tk < 0 || H <= 0 || Hkv <= 0 || H % Hkv || (hd != 64 && hd != 128 && hd != 256)) return 0;
    int splits, chunk;
    decode_plan(B, Lq, Tk, H, Hkv, &splits, &chunk);
    return (size_t)B * H * Lq * splits * (hd + 2) * sizeof(float);
}

attn_status attn_decode(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                        void* workspace, size_t workspace_bytes, int B, int Lq, int Tk, int H, int Hkv, int hd,
                        float scale, int causal, int window, float softcap, int q_offset, const float* key_mask,
                        long long key_mask_bstride, void* stream) {
    attn_status st = check_common(dt, B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride, true);
    if (st != ATTN_OK) return st;
    if (Lq > 16 || (H / Hkv) * Lq > 64) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Lq == 0) return ATTN_OK;
    if (dt == ATTN_F32)  // fp32 stays on the fp32 CUDA-core kernel
        return attn_fwd(dt, q, k, v, o, lse, B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset,
                        key_mask, key_mask_bstride, stream);
    if (!q || !o || (Tk > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (Tk == 0)
        return fill_empty(dt, o, (long long)B * Lq * H * hd, lse, lse ? (long long)B * H * Lq : 0, s);
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd))
        return ATTN_ERR_INVALID_ARG;
    Params p = base_params(B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                           key_mask_bstride);
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.ws = static_cast<float*>(workspace);
    decode_plan(B, Lq, Tk, H, Hkv, &p.splits, &p.chunk);
    DecMaps maps;
    if (!make_map(&maps.k, dt, k, (long long)Hkv * hd, Tk, B, 64) ||
        !make_map(&maps.v, dt, v, (long long)Hkv * hd, Tk, B, 64))
        return ATTN_ERR_CUDA;
    return counted(launch_decode(p, (int)dt, maps, s), 2);
}

attn_status attn_decode_len(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                            void* workspace, size_t workspace_bytes, int B, int Lq, int Tk, int H, int Hkv,
                            int hd, float scale, int causal, int window, float softcap, const int* lengths,
                            const float* key_mask, long long key_mask_bstride, void* stream) {
    attn_status st = check_common(dt, B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, 0, key_mask,
                                  key_mask_bstride, true);
    if (st != ATTN_OK) return st;
    if (!lengths || (reinterpret_cast<uintptr_t>(lengths) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (dt == ATTN_F32) return ATTN_ERR_UNSUPPORTED;  // the 16-bit split kernels only
    if (Lq > 16 || (H / Hkv) * Lq > 64) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Lq == 0) return ATTN_OK;
    if (!q || !o || (Tk > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (Tk == 0)
        return fill_empty(dt, o, (long long)B * Lq * H * hd, lse, lse ? (long long)B * H * Lq : 0, s);
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd))
        return ATTN_ERR_INVALID_ARG;
    Params p = base_params(B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, 0, key_mask,
                           key_mask_bstride);
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.ws = static_cast<float*>(workspace);
    p.lengths = lengths;
    // the plan depends on the capacity only, so a captured launch stays valid as lengths change
    decode_plan(B, Lq, Tk, H, Hkv, &p.splits, &p.chunk);
    DecMaps maps;
    if (!make_map(&maps.k, dt, k, (long long)Hkv * hd, Tk, B, 64) ||
        !make_map(&maps.v, dt, v, (long long)Hkv * hd, Tk, B, 64))
        return ATTN_ERR_CUDA;
    return counted(launch_decode(p, (int)dt, maps, s), 2);
}


attn_status attn_decode_noalloc(attn_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int Lq, int Tk, int H, int Hkv, int hd, float scale, int causal, int window,
                                float softcap, int q_offset, const float* key_mask, long long key_mask_bstride,
                                void* stream) {
    attn_status st = check_common(dt, B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                                  key_mask_bstride, true);
    if (st != ATTN_OK) return st;
    if (Lq > 16 || (H / Hkv) * Lq > 64) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || Lq == 0) return ATTN_OK;
    if (dt == ATTN_F32)  // the fp32 forward kernel needs no scratch
        return attn_fwd(dt, q, k, v, o, lse, B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset,
                        key_mask, key_mask_bstride, stream);
    if (!q || !o || (Tk > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (Tk == 0)
        return fill_empty(dt, o, (long long)B * Lq * H * hd, lse, lse ? (long long)B * H * Lq : 0, s);
    if (attn_decode_workspace_size(B, Lq, Tk, H, Hkv, hd) > kDecodeScratchBytes) return ATTN_ERR_UNSUPPORTED;
    float* scratch = nullptr;
    if (decode_noalloc_scratch(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
    Params p = base_params(B, Lq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset, key_mask,
                           key_mask_bstride);
    if (!p.status) return ATTN_ERR_CUDA;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.ws = scratch;
    decode_plan(B, Lq, Tk, H, Hkv, &p.splits, &p.chunk);
    DecMaps maps;
    if (!make_map(&maps.k, dt, k, (long long)Hkv * hd, Tk, B, 64) ||
        !make_map(&maps.v, dt, v, (long long)Hkv * hd, Tk, B, 64))
        return ATTN_ERR_CUDA;
    return counted(launch_decode(p, (int)dt, maps, s), 2);
}

attn_status attn_get_device_status(void* stream, unsigned int* detail) {
    unsigned int* ptr = status_ptr();
    if (!ptr) return ATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpy(&word, ptr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpy(ptr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
    if (detail) *detail = word;
    if (word & ~(unsigned int)ST_VARLEN_BOUNDS) return ATTN_ERR_TIMEOUT;
    return word ? ATTN_ERR_INVALID_ARG : ATTN_OK;
}

attn_status attn_selftest_bounded_wait(unsigned int timeout_us, void* stream) {
    if (timeout_us == 0 || timeout_us > 2000000u) return ATTN_ERR_INVALID_ARG;
    unsigned int* ptr = status_ptr();
    if (!ptr) return ATTN_ERR_CUDA;
    return counted(launch_selftest_wait(ptr, timeout_us, static_cast<cudaStream_t>(stream)), 1);
}

}  // extern "C"

// --------------------------------------------------- packed fused-QKV rows
namespace {

// The q, k and v columns of a packed [L][3*H*hd] row block copied into three
// contiguous [L][H*hd] tensors (one strided copy each).
attn_status split_qkv(attn_dtype dt, const void* qkv, void* q, void* k, void* v, int L, int H, int hd,
                      cudaStream_t s) {
    const size_t w = (size_t)H * hd * elem_size(dt);
    const uint8_t* src = static_cast<const uint8_t*>(qkv);
    void* dst[3] = {q, k, v};
    for (int t = 0; t < 3; ++t)
        if (cudaMemcpy2DAsync(dst[t], w, src + t * w, 3 * w, w, (size_t)L, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status check_packed(attn_dtype dt, const void* qkv, const int* seq_bounds, int L, int H, int hd, float scale,
                         int window) {
    if (L < 0 || window < 0) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_common(dt, 1, L, L, H, H, hd, scale, 0, 0, 0.f, 0, nullptr, 0);
    if (st != ATTN_OK) return st;
    if (L > 0 && (!qkv || !seq_bounds || !aligned16(qkv) || (reinterpret_cast<uintptr_t>(seq_bounds) & 7u)))
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// One batch of L rows, keys and queries alike, no causal rule; brotensor's
// bidirectional window |r - j| <= window/2 is the two-sided window (window/2, window/2).
Params packed_params(const int* seq_bounds, int L, int H, int hd, float scale, int window) {
    Params p = base_params(1, L, L, H, H, hd, scale, 0, 0, 0.f, 0, nullptr, 0);
    p.wl = p.wr = window > 0 ? window / 2 : -1;
    p.row_bounds = reinterpret_cast<const int2*>(seq_bounds);
    return p;
}

size_t tensor_bytes(attn_dtype dt, int L, int H, int hd) { return align256((size_t)L * H * hd * elem_size(dt)); }

// Heaviest-first orders of the row blocks of a packed batch, for the work-item
// numbering of the tensor-core kernels: blocks of 256 rows (the forward's items) into
// ord256, of 128 rows (the dQ items and the dK/dV key blocks) into ord128.  A block's
// weight is the span of keys its rows see, from its first row's sequence start (less
// the window) to its last row's sequence end (plus the window); with the bounds
// monotone down the rows, that span holds all of the block's visible pairs.  Ties keep
// block order.  One CTA, for at most kOrderMax blocks of 128 rows.
constexpr int kOrderMax = 2048;
__device__ __forceinline__ void rank_blocks(const int* cost, int n, int* ord) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int c = cost[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const int cj = cost[j];
            rank += (cj > c || (cj == c && j < i)) ? 1 : 0;
        }
        ord[rank] = i;
    }
}
__global__ void packed_order_kernel(const int2* sb, int L, int wl, int wr, int* ord256, int* ord128) {
    // sequence start of each 128-row block's first row, sequence end of its last row
    __shared__ int lo_s[kOrderMax], hi_s[kOrderMax];
    __shared__ int cost[kOrderMax + kOrderMax / 2];  // 128-row blocks, then 256-row blocks
    const int n128 = (L + 127) / 128, n256 = (L + 255) / 256;
    for (int i = threadIdx.x; i < n128; i += blockDim.x) {
        lo_s[i] = min(max(__ldg(&sb[i * 128].x), 0), L);
        hi_s[i] = min(max(__ldg(&sb[min(i * 128 + 128, L) - 1].y), 0), L);
    }
    __syncthreads();
    // the span of keys rows r0 .. r1 see: 128-row blocks b0 .. b1
    auto span = [&](int b0, int b1, int r0, int r1) {
        int lo = lo_s[b0], hi = hi_s[b1];
        if (wl >= 0) lo = max(lo, r0 - wl);
        if (wr >= 0) hi = min(hi, r1 + wr + 1);
        return max(hi - lo, 0);
    };
    for (int i = threadIdx.x; i < n128 + n256; i += blockDim.x) {
        if (i < n128) {
            cost[i] = span(i, i, i * 128, min(i * 128 + 128, L) - 1);
        } else {
            const int k = i - n128;
            cost[i] = span(2 * k, min(2 * k + 1, n128 - 1), k * 256, min(k * 256 + 256, L) - 1);
        }
    }
    __syncthreads();
    rank_blocks(cost, n128, ord128);
    rank_blocks(cost + n128, n256, ord256);
}

// The two orders in the workspace at ws (ints: ord256 then ord128), or false when the
// batch has too many blocks (the kernels then keep their plain order).
bool packed_order(const int* seq_bounds, int L, const Params& p, void* ws, int** ord256, int** ord128,
                  cudaStream_t s, attn_status* st) {
    const int n256 = (L + 255) / 256, n128 = (L + 127) / 128;
    *ord256 = *ord128 = nullptr;
    *st = ATTN_OK;
    if (n128 > kOrderMax) return false;
    int* o = static_cast<int*>(ws);
    packed_order_kernel<<<1, 1024, 0, s>>>(reinterpret_cast<const int2*>(seq_bounds), L, p.wl, p.wr, o, o + n256);
    if ((*st = counted(cudaGetLastError(), 1)) != ATTN_OK) return false;
    *ord256 = o;
    *ord128 = o + n256;
    return true;
}

// 16-bit rows at hd 64 / 128 go to the tensor-core kernels, whose tensor maps read q,
// k and v in place from the packed rows (and write dq, dk, dv into them); the
// CUDA-core kernels take contiguous copies.
bool packed_in_place(attn_dtype dt, int hd) { return dt != ATTN_F32 && (hd == 64 || hd == 128); }

}  // namespace

extern "C" {

size_t attn_packed_qkv_workspace_size(attn_dtype dt, int L, int H, int hd, int backward) {
    if (L < 0 || H <= 0 || hd <= 0) return 0;
    const size_t t = tensor_bytes(dt, L, H, hd);
    if (!backward) return 3 * t;  // q, k, v
    // q, k, v, O, LSE, dq, dk, dv and the backward's own workspace
    return 7 * t + align256((size_t)H * L * sizeof(float)) + align256(attn_bwd_workspace_size(1, L, H));
}

attn_status attn_packed_qkv_fwd(attn_dtype dt, const void* qkv, const int* seq_bounds, void* o, float* lse,
                                void* workspace, size_t workspace_bytes, int L, int H, int hd, float scale,
                                int window, void* stream) {
    attn_status st = check_packed(dt, qkv, seq_bounds, L, H, hd, scale, window);
    if (st != ATTN_OK) return st;
    if (L == 0) return ATTN_OK;
    if (!o || !workspace || !aligned16(workspace) || workspace_bytes < attn_packed_qkv_workspace_size(dt, L, H, hd, 0))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Params p = packed_params(seq_bounds, L, H, hd, scale, window);
    if (packed_in_place(dt, hd)) {
        const size_t w = (size_t)H * hd * elem_size(dt);
        const uint8_t* r = static_cast<const uint8_t*>(qkv);
        int *ord256, *ord128;
        packed_order(seq_bounds, L, p, workspace, &ord256, &ord128, s, &st);
        if (st != ATTN_OK) return st;
        p.item_order = ord256;
        return fwd_launch(dt, r, r + w, r + 2 * w, o, lse, p, stream, 3LL * H * hd);
    }
    const size_t t = tensor_bytes(dt, L, H, hd);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if ((st = split_qkv(dt, qkv, ws, ws + t, ws + 2 * t, L, H, hd, s)) != ATTN_OK) return st;
    return fwd_launch(dt, ws, ws + t, ws + 2 * t, o, lse, p, stream);
}

attn_status attn_packed_qkv_bwd(attn_dtype dt, const void* qkv, const void* dout, const int* seq_bounds, void* dqkv,
                                void* workspace, size_t workspace_bytes, int L, int H, int hd, float scale,
                                int window, void* stream) {
    attn_status st = check_packed(dt, qkv, seq_bounds, L, H, hd, scale, window);
    if (st != ATTN_OK) return st;
    if (L == 0) return ATTN_OK;
    if (!dout || !dqkv || !aligned16(dout) || !aligned16(dqkv) || !workspace || !aligned16(workspace) ||
        workspace_bytes < attn_packed_qkv_workspace_size(dt, L, H, hd, 1))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t t = tensor_bytes(dt, L, H, hd), lse_bytes = align256((size_t)H * L * sizeof(float));
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t *q = ws, *k = ws + t, *v = ws + 2 * t, *o = ws + 3 * t;
    float* lse = reinterpret_cast<float*>(ws + 4 * t);
    uint8_t *dq = ws + 4 * t + lse_bytes, *dk = dq + t, *dv = dq + 2 * t, *wb = dq + 3 * t;
    const Params p = packed_params(seq_bounds, L, H, hd, scale, window);
    const size_t w = (size_t)H * hd * elem_size(dt);
    // the backward consumes no forward results: O and LSE are formed again here
    if (packed_in_place(dt, hd)) {
        const uint8_t* r = static_cast<const uint8_t*>(qkv);
        uint8_t* g = static_cast<uint8_t*>(dqkv);
        const long long rs = 3LL * H * hd;
        // the block orders go where the CUDA-core path keeps its copy of q
        int *ord256, *ord128;
        packed_order(seq_bounds, L, p, q, &ord256, &ord128, s, &st);
        if (st != ATTN_OK) return st;
        Params pf = p, pb = p;
        pf.item_order = ord256;
        pb.item_order = ord128;
        if ((st = fwd_launch(dt, r, r + w, r + 2 * w, o, lse, pf, stream, rs)) != ATTN_OK) return st;
        return bwd_launch(dt, r, r + w, r + 2 * w, o, dout, lse, g, g + w, g + 2 * w, wb, attn_bwd_workspace_size(1, L, H),
                          pb, stream, 7, rs, rs);
    }
    if ((st = split_qkv(dt, qkv, q, k, v, L, H, hd, s)) != ATTN_OK) return st;
    if ((st = fwd_launch(dt, q, k, v, o, lse, p, stream)) != ATTN_OK) return st;
    if ((st = bwd_launch(dt, q, k, v, o, dout, lse, dq, dk, dv, wb, attn_bwd_workspace_size(1, L, H), p, stream, 7)) !=
        ATTN_OK)
        return st;
    // dq, dk, dv into their columns of the packed gradient rows
    const void* src[3] = {dq, dk, dv};
    for (int c = 0; c < 3; ++c)
        if (cudaMemcpy2DAsync(static_cast<uint8_t*>(dqkv) + c * w, 3 * w, src[c], w, w, (size_t)L,
                              cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return ATTN_ERR_CUDA;
    return ATTN_OK;
}

}  // extern "C"
