// rope.cu -- rotate-half rotary embedding, applied before attention (in place, or
// into another buffer), and the cosine/sine table the forward's fused rotation reads.
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

// grid.x: blocks of blockDim.y tokens; threadIdx.x: pair index / 2.  Reads src and
// writes dst (the same array for the in-place pass); sgn = -1 turns the other way.
template <typename T>
__global__ void rope_kernel(const T* src, T* dst, long long tokens, int T_, int H, int hd, int pos, float sgn,
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
    s0 *= sgn;
    s1 *= sgn;
    const typename P2::V* irow = reinterpret_cast<const typename P2::V*>(src + tok * (long long)H * hd);
    typename P2::V* orow = reinterpret_cast<typename P2::V*>(dst + tok * (long long)H * hd);
    const int h1 = min(H, (int)(blockIdx.y + 1) * kHeadsPerThread);
#pragma unroll 4
    for (int h = blockIdx.y * kHeadsPerThread; h < h1; ++h) {
        const int lo = (h * hd + i) / 2, hi = (h * hd + i + half) / 2;
        const float2 a = P2::to_f2(irow[lo]), b = P2::to_f2(irow[hi]);
        float2 ra, rb;
        rope_turn(a.x, b.x, c0, s0, ra.x, rb.x);
        rope_turn(a.y, b.y, c1, s1, ra.y, rb.y);
        orow[lo] = P2::from_f2(ra);
        orow[hi] = P2::from_f2(rb);
    }
}

// The same with 16-byte accesses: a thread owns VEC consecutive pairs indices i0 ..
// (used when hd/2 is a multiple of VEC, so both halves stay 16-byte aligned).
template <typename T>
__global__ void rope_vec_kernel(const T* src, T* dst, long long tokens, int T_, int H, int hd, int pos, float sgn,
                                const __grid_constant__ RopeFreqs fr) {
    using P2 = Pair2<T>;
    constexpr int VEC = 16 / (int)sizeof(T);
    const long long tok = (long long)blockIdx.x * blockDim.y + threadIdx.y;
    const int i0 = VEC * threadIdx.x, half = hd / 2;
    if (tok >= tokens || i0 >= half) return;
    const double p = (double)pos + (int)(tok % T_);
    float sn[VEC], cs[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        pair_sincos<T>(p, fr.inv_freq[i0 + e], &sn[e], &cs[e]);
        sn[e] *= sgn;
    }
    const T* irow = src + tok * (long long)H * hd;
    T* orow = dst + tok * (long long)H * hd;
    const int h1 = min(H, (int)(blockIdx.y + 1) * kHeadsPerThread);
#pragma unroll 2
    for (int h = blockIdx.y * kHeadsPerThread; h < h1; ++h) {
        union U {
            uint4 u;
            typename P2::V v[VEC / 2];
        } ua, ub;
        ua.u = *reinterpret_cast<const uint4*>(irow + h * hd + i0);
        ub.u = *reinterpret_cast<const uint4*>(irow + h * hd + i0 + half);
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
            const float2 a = P2::to_f2(ua.v[e]), b = P2::to_f2(ub.v[e]);
            float2 ra, rb;
            rope_turn(a.x, b.x, cs[2 * e], sn[2 * e], ra.x, rb.x);
            rope_turn(a.y, b.y, cs[2 * e + 1], sn[2 * e + 1], ra.y, rb.y);
            ua.v[e] = P2::from_f2(ra);
            ub.v[e] = P2::from_f2(rb);
        }
        *reinterpret_cast<uint4*>(orow + h * hd + i0) = ua.u;
        *reinterpret_cast<uint4*>(orow + h * hd + i0 + half) = ub.u;
    }
}

// Cosine and sine of rotary position s (angle (pos + s) * theta^(-2c/hd)) for every
// pair index c < hd/2: tab[2 * (c * npos + s)] = cos, [+1] = sin (consecutive
// positions adjacent, so that threads holding consecutive rows read one line); the
// angle is formed exactly as the 16-bit pass forms it, so that a table-driven turn
// equals that pass.
__global__ void rope_table_kernel(float* tab, int npos, int half, int pos, const __grid_constant__ RopeFreqs fr) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (long long)npos * half) return;
    const int c = (int)(e / npos), s = (int)(e % npos);
    float sn, cs;
    pair_sincos<__half>((double)pos + s, fr.inv_freq[c], &sn, &cs);
    tab[2 * e] = cs;
    tab[2 * e + 1] = sn;
}

RopeFreqs freqs(int hd, double theta) {
    RopeFreqs fr;
    for (int i = 0; i < hd / 2; ++i) fr.inv_freq[i] = pow(theta, -2.0 * i / hd);
    return fr;
}

template <typename T>
cudaError_t rope_typed(const void* src, void* dst, int B, int T_, int H, int hd, int pos, double theta, float sgn,
                       cudaStream_t st) {
    const RopeFreqs fr = freqs(hd, theta);
    const long long tokens = (long long)B * T_;
    constexpr int VEC = 16 / (int)sizeof(T);
    if ((hd / 2) % VEC == 0) {
        const dim3 block(hd / 2 / VEC, 256 / (hd / 2 / VEC));
        const dim3 grid((unsigned)((tokens + block.y - 1) / block.y), (H + kHeadsPerThread - 1) / kHeadsPerThread);
        rope_vec_kernel<T><<<grid, block, 0, st>>>(static_cast<const T*>(src), static_cast<T*>(dst), tokens, T_, H,
                                                    hd, pos, sgn, fr);
    } else {
        const dim3 block(hd / 4, 256 / (hd / 4));
        const dim3 grid((unsigned)((tokens + block.y - 1) / block.y), (H + kHeadsPerThread - 1) / kHeadsPerThread);
        rope_kernel<T><<<grid, block, 0, st>>>(static_cast<const T*>(src), static_cast<T*>(dst), tokens, T_, H, hd,
                                               pos, sgn, fr);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(const void* src, void* dst, int dt, int B, int T_, int H, int hd, int pos, double theta,
                        bool inverse, cudaStream_t s) {
    const float sgn = inverse ? -1.f : 1.f;
    if (dt == 0) return rope_typed<float>(src, dst, B, T_, H, hd, pos, theta, sgn, s);
    if (dt == 1) return rope_typed<__half>(src, dst, B, T_, H, hd, pos, theta, sgn, s);
    return rope_typed<__nv_bfloat16>(src, dst, B, T_, H, hd, pos, theta, sgn, s);
}

cudaError_t launch_rope_table(float* tab, int npos, int hd, int pos, double theta, cudaStream_t s) {
    const long long n = (long long)npos * (hd / 2);
    if (n == 0) return cudaSuccess;
    rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(tab, npos, hd / 2, pos, freqs(hd, theta));
    return cudaGetLastError();
}

}  // namespace attn
