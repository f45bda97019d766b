// rope.cu -- rotate-half rotary embedding, applied in place before attention.
//
// Source: ferrotensor engine/attention.rs, rope / rope_theta: every head vector
// of token s (counted within its sequence) gets position pos + s, and its pair
// (x[i], x[i + hd/2]), i < hd/2, turns by (pos + s) * theta^(-2i/hd).
//
// HBM-bound: each element is read and written once.  A thread owns the pairs
// i, i+1 of one token for every head (two-element loads at i and i + hd/2),
// so the angle -- the only part that needs care -- is formed once per token
// and frequency: the product (pos + s) * theta^(-2i/hd) and its reduction
// modulo 2 pi are done in fp64 (the frequencies come from the host in fp64),
// then sincosf on the reduced angle, so that the rotation keeps fp32 accuracy
// at every position.
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
    rot_sincos(p * fr.inv_freq[i], &s0, &c0);
    rot_sincos(p * fr.inv_freq[i + 1], &s1, &c1);
    typename P2::V* row = reinterpret_cast<typename P2::V*>(x + tok * (long long)H * hd);
#pragma unroll 4
    for (int h = 0; h < H; ++h) {
        typename P2::V* lo = row + (h * hd + i) / 2;
        typename P2::V* hi = row + (h * hd + i + half) / 2;
        const float2 a = P2::to_f2(*lo), b = P2::to_f2(*hi);
        *lo = P2::from_f2(make_float2(a.x * c0 - b.x * s0, a.y * c1 - b.y * s1));
        *hi = P2::from_f2(make_float2(b.x * c0 + a.x * s0, b.y * c1 + a.y * s1));
    }
}

template <typename T>
cudaError_t rope_typed(void* x, int B, int T_, int H, int hd, int pos, double theta, cudaStream_t st) {
    RopeFreqs fr;
    for (int i = 0; i < hd / 2; ++i) fr.inv_freq[i] = pow(theta, -2.0 * i / hd);
    const long long tokens = (long long)B * T_;
    const dim3 block(hd / 4, 256 / (hd / 4));
    const long long blocks = (tokens + block.y - 1) / block.y;
    rope_kernel<T><<<(unsigned)blocks, block, 0, st>>>(static_cast<T*>(x), tokens, T_, H, hd, pos, fr);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(void* x, int dt, int B, int T_, int H, int hd, int pos, double theta, cudaStream_t s) {
    if (dt == 0) return rope_typed<float>(x, B, T_, H, hd, pos, theta, s);
    if (dt == 1) return rope_typed<__half>(x, B, T_, H, hd, pos, theta, s);
    return rope_typed<__nv_bfloat16>(x, B, T_, H, hd, pos, theta, s);
}

}  // namespace attn
