// simt.cu -- CUDA-core attention kernels: the fp32 forward and backward.
//
// fp32 inputs must stay off the tensor cores to keep fp32 accuracy (no TF32,
// no 16-bit P), so these kernels do the whole computation with fp32 FMAs and
// the accurate expf / logf / tanhf.  The same templates also instantiate for
// 16-bit inputs (converted to fp32 on load); the D = rowsum(dO*O) preprocess
// is shared with the tensor-core backward.
//
// Work split (one warp per output row, 8 rows per CTA sharing staged tiles):
//   forward, dQ : CTA = 8 query rows of one (b, h); K/V tiles of 64 keys are
//                 staged in shared memory as fp32, each lane scores 2 keys,
//                 then owns hd/32 output columns for the P.V (or dS.K) update.
//   dK/dV       : CTA = 8 key rows of one (b, kv head); Q/dO tiles of 64 rows
//                 of every query head in the group are staged, each lane
//                 handles 2 query rows; no atomics (the GQA group sum stays in
//                 registers).
// Sources: vision_rs flash_attn2.rs, Forward / Backward - dQ / Backward - dK,dV
// (online-softmax recurrence, p = exp(s - LSE), dS = p (dO.V - D)); forge
// attention.metal, attention_bwd_d_f32 / attention_bwd_dq_f32 /
// attention_bwd_dkv_f32 (D = dO.O, softcap derivative, group sums).
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kRows = 8;   // warps (rows) per CTA
constexpr int kTile = 64;  // keys (or queries) staged per tile

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// capped score in natural units
__device__ __forceinline__ float capped(float s, float softcap) {
    return softcap > 0.f ? softcap * tanhf(s / softcap) : s;
}
// additive score bias of (b, h, i, j), or 0
__device__ __forceinline__ float bias_at(const Params& P, int b, int h, int i, int j) {
    return P.bias ? P.bias[(long long)b * P.bias_sb + (long long)h * P.bias_sh + (long long)i * P.bias_sq +
                           (long long)j * P.bias_sk]
                  : 0.f;
}

// head h of query row i (key row j) of sequence sq
__device__ __forceinline__ long long qoff(const Params& P, const Seq& sq, int i, int h) {
    return ((long long)sq.zb * P.Tq + sq.q0 + i) * (long long)P.H * P.hd + (long long)h * P.hd;
}
__device__ __forceinline__ long long kvoff(const Params& P, const Seq& sq, int j, int kvh) {
    return ((long long)sq.zb * P.Tk + sq.k0 + j) * (long long)P.Hkv * P.hd + (long long)kvh * P.hd;
}
template <typename T>
__device__ __forceinline__ const T* qrow(const Params& P, const void* base, const Seq& sq, int i, int h) {
    return reinterpret_cast<const T*>(base) + qoff(P, sq, i, h);
}
template <typename T>
__device__ __forceinline__ const T* kvrow(const Params& P, const void* base, const Seq& sq, int j, int kvh) {
    return reinterpret_cast<const T*>(base) + kvoff(P, sq, j, kvh);
}

// ------------------------------------------------------------------ forward
template <typename T, int HD>
__global__ void __launch_bounds__(kRows * 32) simt_fwd_kernel(Params P) {
    extern __shared__ float sm[];
    float* Ks = sm;                          // [kTile][HD+1]
    float* Vs = Ks + kTile * (HD + 1);       // [kTile][HD]
    float* Qs = Vs + kTile * HD;             // [kRows][HD]
    float* Ps = Qs + kRows * HD;             // [kRows][kTile]
    const int b = blockIdx.z, h = blockIdx.y, kvh = h / P.G;
    const Seq sq = seq_any(P, b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kRows;
    if (i0 >= sq.tq) return;  // (packed) past this sequence's rows
    const int i = i0 + warp;
    const bool row_ok = i < sq.tq;
    const int p = i + P.q_offset;
    const int ilast = min(i0 + kRows, sq.tq) - 1;
    int lo, hi;
    key_range(P.wl, P.wr, sq.tk, i0 + P.q_offset, ilast + P.q_offset, &lo, &hi);
    if (P.row_bounds) {  // packed fused-QKV rows: the block's first and last rows bound its keys
        lo = max(lo, row_keys(P, i0, sq.tk).x);
        hi = max(lo, min(hi, row_keys(P, ilast, sq.tk).y));
    }

    for (int d = lane; d < HD; d += 32)
        Qs[warp * HD + d] = row_ok ? Elem<T>::to_f(qrow<T>(P, P.q, sq, i, h)[d]) : 0.f;

    float m = -INFINITY, l = 0.f;
    float acc[HD / 32];
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) acc[c] = 0.f;

    for (int j0 = (lo / kTile) * kTile; j0 < hi; j0 += kTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTile * HD; e += blockDim.x) {
            const int jj = e / HD, d = e % HD, j = j0 + jj;
            float kv = 0.f, vv = 0.f;
            if (j < sq.tk) {
                kv = Elem<T>::to_f(kvrow<T>(P, P.k, sq, j, kvh)[d]);
                vv = Elem<T>::to_f(kvrow<T>(P, P.v, sq, j, kvh)[d]);
            }
            Ks[jj * (HD + 1) + d] = kv;
            Vs[jj * HD + d] = vv;
        }
        __syncthreads();
        float s[2];
        bool vis[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int jj = lane + 32 * t, j = j0 + jj;
            float dot = 0.f;
#pragma unroll 8
            for (int d = 0; d < HD; ++d) dot = fmaf(Qs[warp * HD + d], Ks[jj * (HD + 1) + d], dot);
            vis[t] = row_ok && visible(P, b, p, j, sq.tk);
            s[t] = vis[t] ? capped(dot * P.scale, P.softcap) + bias_at(P, b, h, i, j) : -INFINITY;
        }
        const float m_new = fmaxf(m, warp_max(fmaxf(s[0], s[1])));
        if (m_new == -INFINITY) continue;  // nothing visible yet for this row (warp-uniform)
        const float alpha = expf(m - m_new);  // 0 when m = -inf
        float pr[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) pr[t] = vis[t] ? expf(s[t] - m_new) : 0.f;
        l = l * alpha + warp_sum(pr[0] + pr[1]);
        Ps[warp * kTile + lane] = pr[0];
        Ps[warp * kTile + lane + 32] = pr[1];
        __syncwarp();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
            float a = acc[c] * alpha;
            const int d = lane + 32 * c;
#pragma unroll 8
            for (int jj = 0; jj < kTile; ++jj) a = fmaf(Ps[warp * kTile + jj], Vs[jj * HD + d], a);
            acc[c] = a;
        }
        __syncwarp();
        m = m_new;
    }
    if (!row_ok) return;
    T* orow = reinterpret_cast<T*>(P.o) + qoff(P, sq, i, h);
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) orow[lane + 32 * c] = Elem<T>::from_f(acc[c] * inv);
    if (P.lse && lane == 0)
        P.lse[((long long)b * P.H + h) * P.Tq + i] = l > 0.f ? m + logf(l) : -INFINITY;
}

// ------------------------------------------------------- backward: D = dO.O
// D = dO.O and LSE*log2(e) for every (b, i, h) row, i < tq_pad, into the padded
// [B*H][tq_pad] workspace rows (padding rows get D = 0, LSE = +inf so they
// contribute nothing).  HBM-bound: each thread reads 16 bytes of O and of dO,
// LPR = hd*sizeof(T)/16 lanes share a row, rows in (b, i, h) order so
// consecutive lanes read consecutive memory.
template <typename T, int LPR>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(Params P) {
    constexpr int V = 16 / (int)sizeof(T);  // elements per 16-byte load
    const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = gt / LPR;
    const int sub = (int)(gt % LPR);
    const long long rows = (long long)P.B * P.tq_pad * P.H;
    const bool live = row < rows;
    const int h = live ? (int)(row % P.H) : 0;
    const long long bi = live ? row / P.H : 0;
    const int i = (int)(bi % P.tq_pad), b = (int)(bi / P.tq_pad);
    const Seq sq = seq_any(P, live ? b : 0);
    float acc = 0.f;
    if (live && i < sq.tq) {
        const uint4 ov = reinterpret_cast<const uint4*>(qrow<T>(P, P.o_in, sq, i, h))[sub];
        const uint4 gv = reinterpret_cast<const uint4*>(qrow<T>(P, P.dout, sq, i, h))[sub];
        const T* oe = reinterpret_cast<const T*>(&ov);
        const T* ge = reinterpret_cast<const T*>(&gv);
#pragma unroll
        for (int e = 0; e < V; ++e) acc = fmaf(Elem<T>::to_f(oe[e]), Elem<T>::to_f(ge[e]), acc);
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, LPR);
    if (!live || sub != 0) return;
    const long long srow = ((long long)b * P.H + h) * P.tq_pad + i;
    if (i >= sq.tq) {
        P.ndelta[srow] = 0.f;
        P.nlse2[srow] = -INFINITY;
        return;
    }
    P.ndelta[srow] = -acc;
    const float l = P.lse_in[((long long)b * P.H + h) * P.Tq + i];
    P.nlse2[srow] = l == -INFINITY ? -INFINITY : -l * 1.4426950408889634f;
}

// -------------------------------------------------------------- backward: dQ
template <typename T, int HD>
__global__ void __launch_bounds__(kRows * 32) simt_dq_kernel(Params P) {
    extern __shared__ float sm[];
    float* Ks = sm;                      // [kTile][HD+1]
    float* Vs = Ks + kTile * (HD + 1);   // [kTile][HD+1]
    float* Qs = Vs + kTile * (HD + 1);   // [kRows][HD]
    float* Gs = Qs + kRows * HD;         // [kRows][HD]  dO
    float* Ss = Gs + kRows * HD;         // [kRows][kTile] dS
    const int b = blockIdx.z, h = blockIdx.y, kvh = h / P.G;
    const Seq sq = seq_any(P, b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kRows;
    if (i0 >= sq.tq) return;  // (packed) past this sequence's rows
    const int i = i0 + warp;
    const bool row_ok = i < sq.tq;
    const int p = i + P.q_offset;
    const int ilast = min(i0 + kRows, sq.tq) - 1;
    int lo, hi;
    key_range(P.wl, P.wr, sq.tk, i0 + P.q_offset, ilast + P.q_offset, &lo, &hi);
    if (P.row_bounds) {  // packed fused-QKV rows: the block's first and last rows bound its keys
        lo = max(lo, row_keys(P, i0, sq.tk).x);
        hi = max(lo, min(hi, row_keys(P, ilast, sq.tk).y));
    }
    for (int d = lane; d < HD; d += 32) {
        Qs[warp * HD + d] = row_ok ? Elem<T>::to_f(qrow<T>(P, P.q, sq, i, h)[d]) : 0.f;
        Gs[warp * HD + d] = row_ok ? Elem<T>::to_f(qrow<T>(P, P.dout, sq, i, h)[d]) : 0.f;
    }
    const long long srow = ((long long)b * P.H + h) * P.Tq + i;
    const float lse = row_ok ? P.lse_in[srow] : -INFINITY;
    const float Dd = row_ok ? -P.ndelta[((long long)b * P.H + h) * P.tq_pad + i] : 0.f;
    const bool live = row_ok && lse != -INFINITY;
    float acc[HD / 32];
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) acc[c] = 0.f;

    for (int j0 = (lo / kTile) * kTile; j0 < hi; j0 += kTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTile * HD; e += blockDim.x) {
            const int jj = e / HD, d = e % HD, j = j0 + jj;
            float kv = 0.f, vv = 0.f;
            if (j < sq.tk) {
                kv = Elem<T>::to_f(kvrow<T>(P, P.k, sq, j, kvh)[d]);
                vv = Elem<T>::to_f(kvrow<T>(P, P.v, sq, j, kvh)[d]);
            }
            Ks[jj * (HD + 1) + d] = kv;
            Vs[jj * (HD + 1) + d] = vv;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int jj = lane + 32 * t, j = j0 + jj;
            float ds = 0.f;
            if (live && visible(P, b, p, j, sq.tk)) {
                float qk = 0.f, gv = 0.f;
#pragma unroll 8
                for (int d = 0; d < HD; ++d) {
                    qk = fmaf(Qs[warp * HD + d], Ks[jj * (HD + 1) + d], qk);
                    gv = fmaf(Gs[warp * HD + d], Vs[jj * (HD + 1) + d], gv);
                }
                const float s = qk * P.scale;
                float st = s, dcap = 1.f;
                if (P.softcap > 0.f) {
                    const float th = tanhf(s / P.softcap);
                    st = P.softcap * th;
                    dcap = 1.f - th * th;
                }
                const float pr = expf(st + bias_at(P, b, h, i, j) - lse);
                ds = pr * (gv - Dd) * dcap;
            }
            Ss[warp * kTile + jj] = ds;
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
            float a = acc[c];
            const int d = lane + 32 * c;
#pragma unroll 8
            for (int jj = 0; jj < kTile; ++jj) a = fmaf(Ss[warp * kTile + jj], Ks[jj * (HD + 1) + d], a);
            acc[c] = a;
        }
        __syncwarp();
    }
    if (!row_ok) return;
    T* out = reinterpret_cast<T*>(P.dq) + qoff(P, sq, i, h);
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) out[lane + 32 * c] = Elem<T>::from_f(acc[c] * P.scale);
}

// ----------------------------------------------------------- backward: dK/dV
template <typename T, int HD>
__global__ void __launch_bounds__(kRows * 32) simt_dkdv_kernel(Params P) {
    extern __shared__ float sm[];
    float* Qs = sm;                      // [kTile][HD+1]
    float* Gs = Qs + kTile * (HD + 1);   // [kTile][HD+1]  dO
    float* Ks = Gs + kTile * (HD + 1);   // [kRows][HD]
    float* Vs = Ks + kRows * HD;         // [kRows][HD]
    float* Ls = Vs + kRows * HD;         // [kTile] LSE
    float* Ds = Ls + kTile;              // [kTile] D
    float* Pw = Ds + kTile;              // [kRows][kTile] P
    float* Sw = Pw + kRows * kTile;      // [kRows][kTile] dS
    const int b = blockIdx.z, kvh = blockIdx.y;
    const Seq sq = seq_any(P, b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j0 = blockIdx.x * kRows;
    if (j0 >= sq.tk) return;  // (packed) past this sequence's keys
    const int j = j0 + warp;
    const bool key_ok = j < sq.tk;
    const int jlast = min(j0 + kRows, sq.tk);
    int qlo, qhi;
    query_range(P.wl, P.wr, sq.tq, P.q_offset, j0, jlast, &qlo, &qhi);
    if (P.row_bounds) {  // packed fused-QKV rows: a key is seen only from its own sequence
        qlo = max(qlo, row_keys(P, j0, sq.tq).x);
        qhi = max(qlo, min(qhi, row_keys(P, jlast - 1, sq.tq).y));
    }
    for (int d = lane; d < HD; d += 32) {
        Ks[warp * HD + d] = key_ok ? Elem<T>::to_f(kvrow<T>(P, P.k, sq, j, kvh)[d]) : 0.f;
        Vs[warp * HD + d] = key_ok ? Elem<T>::to_f(kvrow<T>(P, P.v, sq, j, kvh)[d]) : 0.f;
    }
    float dk[HD / 32], dv[HD / 32];
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) dk[c] = dv[c] = 0.f;

    for (int h = kvh * P.G; h < (kvh + 1) * P.G; ++h) {
        for (int i0 = (qlo / kTile) * kTile; i0 < qhi; i0 += kTile) {
            __syncthreads();
            for (int e = threadIdx.x; e < kTile * HD; e += blockDim.x) {
                const int ii = e / HD, d = e % HD, i = i0 + ii;
                float qv = 0.f, gv = 0.f;
                if (i < sq.tq) {
                    qv = Elem<T>::to_f(qrow<T>(P, P.q, sq, i, h)[d]);
                    gv = Elem<T>::to_f(qrow<T>(P, P.dout, sq, i, h)[d]);
                }
                Qs[ii * (HD + 1) + d] = qv;
                Gs[ii * (HD + 1) + d] = gv;
            }
            for (int ii = threadIdx.x; ii < kTile; ii += blockDim.x) {
                const int i = i0 + ii;
                const long long srow = ((long long)b * P.H + h) * P.Tq + i;
                Ls[ii] = i < sq.tq ? P.lse_in[srow] : -INFINITY;
                Ds[ii] = i < sq.tq ? -P.ndelta[((long long)b * P.H + h) * P.tq_pad + i] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int ii = lane + 32 * t, i = i0 + ii;
                float pr = 0.f, ds = 0.f;
                if (key_ok && i < sq.tq && Ls[ii] != -INFINITY && visible(P, b, i + P.q_offset, j, sq.tk)) {
                    float qk = 0.f, gv = 0.f;
#pragma unroll 8
                    for (int d = 0; d < HD; ++d) {
                        qk = fmaf(Qs[ii * (HD + 1) + d], Ks[warp * HD + d], qk);
                        gv = fmaf(Gs[ii * (HD + 1) + d], Vs[warp * HD + d], gv);
                    }
                    const float s = qk * P.scale;
                    float st = s, dcap = 1.f;
                    if (P.softcap > 0.f) {
                        const float th = tanhf(s / P.softcap);
                        st = P.softcap * th;
                        dcap = 1.f - th * th;
                    }
                    pr = expf(st + bias_at(P, b, h, i, j) - Ls[ii]);
                    ds = pr * (gv - Ds[ii]) * dcap;
                }
                Pw[warp * kTile + ii] = pr;
                Sw[warp * kTile + ii] = ds;
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                const int d = lane + 32 * c;
                float a = dv[c], g = dk[c];
#pragma unroll 8
                for (int ii = 0; ii < kTile; ++ii) {
                    a = fmaf(Pw[warp * kTile + ii], Gs[ii * (HD + 1) + d], a);
                    g = fmaf(Sw[warp * kTile + ii], Qs[ii * (HD + 1) + d], g);
                }
                dv[c] = a;
                dk[c] = g;
            }
            __syncwarp();
        }
    }
    if (!key_ok) return;
    const long long off = kvoff(P, sq, j, kvh);
    T* dkp = reinterpret_cast<T*>(P.dk) + off;
    T* dvp = reinterpret_cast<T*>(P.dv) + off;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
        dkp[lane + 32 * c] = Elem<T>::from_f(dk[c] * P.scale);
        dvp[lane + 32 * c] = Elem<T>::from_f(dv[c]);
    }
}

template <typename T, int HD>
cudaError_t fwd_typed(const Params& p, cudaStream_t s) {
    const size_t smem = sizeof(float) * (kTile * (HD + 1) + kTile * HD + kRows * HD + kRows * kTile);
    auto kern = simt_fwd_kernel<T, HD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Tq + kRows - 1) / kRows, p.H, p.B);
    kern<<<grid, kRows * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T, int LPR>
cudaError_t preprocess_launch(const Params& p, cudaStream_t s) {
    const long long threads = (long long)p.B * p.tq_pad * p.H * LPR;
    const int block = 256;
    bwd_preprocess_kernel<T, LPR><<<(unsigned)((threads + block - 1) / block), block, 0, s>>>(p);
    return cudaGetLastError();
}

// The same D pass for any head size: one warp per (b, i, h) row, lanes striding
// over its hd elements.
template <typename T>
__global__ void __launch_bounds__(256) bwd_preprocess_any_kernel(Params P) {
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)P.B * P.tq_pad * P.H;
    if (row >= rows) return;  // whole warps leave together
    const int h = (int)(row % P.H);
    const long long bi = row / P.H;
    const int i = (int)(bi % P.tq_pad), b = (int)(bi / P.tq_pad);
    const Seq sq = seq_any(P, b);
    float acc = 0.f;
    if (i < sq.tq) {
        const T* o = qrow<T>(P, P.o_in, sq, i, h);
        const T* g = qrow<T>(P, P.dout, sq, i, h);
        for (int d = lane; d < P.hd; d += 32) acc = fmaf(Elem<T>::to_f(o[d]), Elem<T>::to_f(g[d]), acc);
    }
    acc = warp_sum(acc);
    if (lane != 0) return;
    const long long srow = ((long long)b * P.H + h) * P.tq_pad + i;
    if (i >= sq.tq) {
        P.ndelta[srow] = 0.f;
        P.nlse2[srow] = -INFINITY;
        return;
    }
    P.ndelta[srow] = -acc;
    const float l = P.lse_in[((long long)b * P.H + h) * P.Tq + i];
    P.nlse2[srow] = l == -INFINITY ? -INFINITY : -l * 1.4426950408889634f;
}

template <typename T>
cudaError_t preprocess_typed(const Params& p, cudaStream_t s) {
    // lanes per row = hd * sizeof(T) / 16 for hd 64 or 128 (and 16-bit hd 256: a warp of
    // 16-byte loads per row); a warp per row with element loads otherwise
    const int lpr = p.hd * (int)sizeof(T) / 16;
    if (p.hd == 64 || p.hd == 128 || (p.hd == 256 && sizeof(T) == 2)) {
        if (lpr == 8) return preprocess_launch<T, 8>(p, s);
        if (lpr == 16) return preprocess_launch<T, 16>(p, s);
        return preprocess_launch<T, 32>(p, s);
    }
    const long long threads = (long long)p.B * p.tq_pad * p.H * 32;
    bwd_preprocess_any_kernel<T><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T, int HD>
cudaError_t bwd_typed(const Params& p, int phases, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    // (packed sequences: a zero bound leaves nothing to launch for that pass)
    if ((phases & 1) && p.tq_pad > 0) {
        e = preprocess_typed<T>(p, s);
        if (e != cudaSuccess) return e;
    }
    if ((phases & 2) && p.Tk > 0) {
        const size_t smem_kv =
            sizeof(float) * (2 * kTile * (HD + 1) + 2 * kRows * HD + 2 * kTile + 2 * kRows * kTile);
        auto kkv = simt_dkdv_kernel<T, HD>;
        e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv);
        if (e != cudaSuccess) return e;
        kkv<<<dim3((p.Tk + kRows - 1) / kRows, p.Hkv, p.B), kRows * 32, smem_kv, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (!(phases & 4) || p.Tq == 0) return cudaSuccess;
    const size_t smem_dq =
        sizeof(float) * (2 * kTile * (HD + 1) + 2 * kRows * HD + kRows * kTile);
    auto kdq = simt_dq_kernel<T, HD>;
    e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dq);
    if (e != cudaSuccess) return e;
    kdq<<<dim3((p.Tq + kRows - 1) / kRows, p.H, p.B), kRows * 32, smem_dq, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

template <int HD>
cudaError_t fwd_hd(const Params& p, int dt, cudaStream_t s) {
    if (dt == 0) return fwd_typed<float, HD>(p, s);
    if (dt == 1) return fwd_typed<__half, HD>(p, s);
    return fwd_typed<__nv_bfloat16, HD>(p, s);
}
template <int HD>
cudaError_t bwd_hd(const Params& p, int dt, int phases, cudaStream_t s) {
    if (dt == 0) return bwd_typed<float, HD>(p, phases, s);
    if (dt == 1) return bwd_typed<__half, HD>(p, phases, s);
    return bwd_typed<__nv_bfloat16, HD>(p, phases, s);
}

// head sizes 32, 64, 96, 128, 256 (the caller has checked)
cudaError_t launch_simt_fwd(const Params& p, int dt, cudaStream_t s) {
    switch (p.hd) {
        case 32: return fwd_hd<32>(p, dt, s);
        case 64: return fwd_hd<64>(p, dt, s);
        case 96: return fwd_hd<96>(p, dt, s);
        case 128: return fwd_hd<128>(p, dt, s);
        default: return fwd_hd<256>(p, dt, s);
    }
}

cudaError_t launch_bwd_preprocess(const Params& p, int dt, cudaStream_t s) {
    if (dt == 0) return preprocess_typed<float>(p, s);
    if (dt == 1) return preprocess_typed<__half>(p, s);
    return preprocess_typed<__nv_bfloat16>(p, s);
}

cudaError_t launch_simt_bwd(const Params& p, int dt, int phases, cudaStream_t s) {
    switch (p.hd) {
        case 32: return bwd_hd<32>(p, dt, phases, s);
        case 64: return bwd_hd<64>(p, dt, phases, s);
        case 96: return bwd_hd<96>(p, dt, phases, s);
        case 128: return bwd_hd<128>(p, dt, phases, s);
        default: return bwd_hd<256>(p, dt, phases, s);
    }
}

}  // namespace attn
