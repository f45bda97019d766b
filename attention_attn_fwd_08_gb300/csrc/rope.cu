// rope.cu -- rotate-half rotary embedding, applied in place before attention.
//
// Source: ferrotensor engine/attention.rs, rope / rope_theta: every head vector
// of token s (counted within its sequence) gets position pos + s, and its pair
// (x[i], x[i + hd/2]), i < hd/2, turns by (pos + s) * theta^(-2i/hd).
//
// HBM-bound: each element is read and written once.  A thread owns a few
// consecutive pair indices of one token for a group of heads, so the angle is
// formed once per (token, frequency, head group).  For fp32 data the product
// (pos + s) * theta^(-2i/hd) and its reduction modulo 2 pi are done in fp64
// (the frequencies come from the host in fp64), then sincosf on the reduced
// angle, so that the rotation keeps fp32 accuracy at every position; 16-bit
// data takes the fp32 product (its error, below 1e-3 rad at position 10^4,
// stays under the 16-bit rounding of the result) and spares the slow fp64 unit.
#include "kernels.h"

namespace attn {
namespace {

struct RopeFreqs {
    double inv_freq[128];  // theta^(-2i/hd), i < hd/2
};

template <typename T> struct Pair2;
template <> struct Pair2<float> {
    using V = float2;
    static __device__ __forceinline__ float2 to_f2(V v) { return v; }
    static __device__ __forceinline__ V from_f2(float2 f) { return f; }
};
template <> struct Pair2<__half> {
    using V = __half2;
    static __device__ __forceinline__ float2 to_f2(V v) { return __half22float2(v); }
    static __device__ __forceinline__ V from_f2(float2 f) { return __float22half2_rn(f); }
};
template <> struct Pair2<__nv_bfloat16> {
    using V = __nv_bfloat162;
    static __device__ __forceinline__ float2 to_f2(V v) { return __bfloat1622float2(v); }
    static __device__ __forceinline__ V from_f2(float2 f) { return __float22bfloat162_rn(f); }
};

// angle reduced to [-pi, pi] in fp64, then fp32 sine and cosine
__device__ __forceinline__ void rot_sincos(double angle, float* s, float* c) {
    const double kTwoPi = 6.283185307179586;
    const double k = rint(angle * (1.0 / kTwoPi));
    const float r = (float)fma(-k, kTwoPi, angle);
    sincosf(r, s, c);
}
// sine and cosine of p * f for pair index i: fp64 angle for fp32 data, fp32 otherwise
template <typename T>
__device__ __forceinline__ void pair_sincos(double p, double f, float* s, float* c) {
    if constexpr (sizeof(T) == 4) rot_sincos(p * f, s, c);
    else sincosf((float)p * (float)f, s, c);
}
constexpr int kHeadsPerThread = 4;

// grid.x: blocks of blockDim.y tokens; threadIdx.x: pair index / 2
template <typename T>
__global__ void rope_kernel(T* x, long long tokens, int T_, int H, int hd, int pos,
                            const __grid_constant__ RopeFreqs fr) {
    using P2 = Pair2<T>;
    const long long tok = (long long)blockIdx.x * blockDim.y + threadIdx.y;
    const int i = 2 * threadIdx.x, half = hd / 2;
    if (tok >= tokens || i >= half) return;
    const int s = (int)(tok % T_);
    const double p = (double)pos + s;
    float s0, c0, s1, c1;
    pair_sincos<T>(p, fr.inv_freq[i], &s0, &c0);
    pair_sincos<T>(p, fr.inv_freq[i + 1], &s1, &c1);
    typename P2::V* row = reinterpret_cast<typename P2::V*>(x + tok * (long long)H * hd);
    const int h1 = min(H, (int)(blockIdx.y + 1) * kHeadsPerThread);
#pragma unroll 4
    for (int h = blockIdx.y * kHeadsPerThread; h < h1; ++h) {
        typename P2::V* lo = row + (h * hd + i) / 2;
        typename P2::V* hi = row + (h * hd + i + half) / 2;
        const float2 a = P2::to_f2(*lo), b = P2::to_f2(*hi);
        *lo = P2::from_f2(make_float2(a.x * c0 - b.x * s0, a.y * c1 - b.y * s1));
        *hi = P2::from_f2(make_float2(b.x * c0 + a.x * s0, b.y * c1 + a.y * s1));
    }
}

// The same with 16-byte accesses: a thread owns VEC consecutive pairs indices i0 ..
// (used when hd/2 is a multiple of VEC, so both halves stay 16-byte aligned).
template <typename T>
__global__ void rope_vec_kernel(T* x, long long tokens, int T_, int H, int hd, int pos,
                                const __grid_constant__ RopeFreqs fr) {
    using P2 = Pair2<T>;
    constexpr int VEC = 16 / (int)sizeof(T);
    const long long tok = (long long)blockIdx.x * blockDim.y + threadIdx.y;
    const int i0 = VEC * threadIdx.x, half = hd / 2;
    if (tok >= tokens || i0 >= half) return;
    const double p = (double)pos + (int)(tok % T_);
    float sn[VEC], cs[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) pair_sincos<T>(p, fr.inv_freq[i0 + e], &sn[e], &cs[e]);
    T* row = x + tok * (long long)H * hd;
    const int h1 = min(H, (int)(blockIdx.y + 1) * kHeadsPerThread);
#pragma unroll 2
    for (int h = blockIdx.y * kHeadsPerThread; h < h1; ++h) {
        uint4* lo = reinterpret_cast<uint4*>(row + h * hd + i0);
        uint4* hi = reinterpret_cast<uint4*>(row + h * hd + i0 + half);
        union U {
            uint4 u;
            typename P2::V v[VEC / 2];
        } ua, ub;
        ua.u = *lo;
        ub.u = *hi;
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
            const float2 a = P2::to_f2(ua.v[e]), b = P2::to_f2(ub.v[e]);
            const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
            ua.v[e] = P2::from_f2(make_float2(a.x * c0 - b.x * s0, a.y * c1 - b.y * s1));
            ub.v[e] = P2::from_f2(make_float2(b.x * c0 + a.x * s0, b.y * c1 + a.y * s1));
        }
        *lo = ua.u;
        *hi = ub.u;
    }
}

template <typename T>
cudaError_t rope_typed(void* x, int B, int T_, int H, int hd, int pos, double theta, cudaStream_t st) {
    RopeFreqs fr;
    for (int i = 0; i < hd / 2; ++i) fr.inv_freq[i] = pow(theta, -2.0 * i / hd);
    const long long tokens = (long long)B * T_;
    constexpr int VEC = 16 / (int)sizeof(T);
    if ((hd / 2) % VEC == 0) {
        const dim3 block(hd / 2 / VEC, 256 / (hd / 2 / VEC));
        const dim3 grid((unsigned)((tokens + block.y - 1) / block.y), (H + kHeadsPerThread - 1) / kHeadsPerThread);
        rope_vec_kernel<T><<<grid, block, 0, st>>>(static_cast<T*>(x), tokens, T_, H, hd, pos, fr);
    } else {
        const dim3 block(hd / 4, 256 / (hd / 4));
        const dim3 grid((unsigned)((tokens + block.y - 1) / block.y), (H + kHeadsPerThread - 1) / kHeadsPerThread);
        rope_kernel<T><<<grid, block, 0, st>>>(static_cast<T*>(x), tokens, T_, H, hd, pos, fr);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(void* x, int dt, int B, int T_, int H, int hd, int pos, double theta, cudaStream_t s) {
    if (dt == 0) return rope_typed<float>(x, B, T_, H, hd, pos, theta, s);
    if (dt == 1) return rope_typed<__half>(x, B, T_, H, hd, pos, theta, s);
    return rope_typed<__nv_bfloat16>(x, B, T_, H, hd, pos, theta, s);
}

}  // namespace attn
