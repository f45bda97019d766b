// decode.cu -- split-KV decode over a long KV cache (fp16 / bf16, hd 64 / 128).
//
// Sources: brotensor ops/flash_attention.h, flash_attention_decode (query row q
// of an L_q block sits at position valid_len - L_q + q and attends [0, p];
// GQA maps query head h to KV head h/(Hq/Hkv); softcap and window as in the
// Gemma-2 extensions) and flash_attention_decode_len (the work is divided over
// the keys, split points change only the rounding, and an R-row block reads
// each cache row once for all R rows).
//
// Design (HBM-bound: every K/V byte is read exactly once per call):
//   split kernel   grid (splits, B*Hkv*row_chunks), 5 warps.  Warp 4 streams
//                  64-key K and V tiles of one KV head with TMA (128-byte
//                  swizzle) into a 3-stage shared-memory ring; warps 0-3 each
//                  take 16 keys of every tile and compute S = Q K^T and O += P V
//                  for all (H/Hkv)*Lq query rows of the group at once (<= 16
//                  rows per CTA) with mma.sync m16n8k16, online softmax in
//                  registers (exp2 domain).  The four warps merge their
//                  (m, l, O) and the CTA writes one unnormalised partial per row.
//   combine kernel one CTA per query row merges the splits by log-sum-exp.
// Sixteen query rows is the natural M of mma.sync; the tcgen05 minimum (M=64)
// would waste 3/4 of every MMA and the path is bound by HBM, not the MMA rate.
#include <math.h>

#include <mutex>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kKeys = 64;     // keys per tile
constexpr int kStages = 3;    // ring depth
constexpr int kThreads = 160; // 4 consumer warps + 1 producer warp
constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct DecSmem {
    static constexpr int kBoxes = HD / 64;
    static constexpr int kTileBytes = kBoxes * kKeys * 128;         // K (or V) tile
    static constexpr int kRingBytes = kStages * 2 * kTileBytes;
    static constexpr int kMergeBytes = 4 * 16 * HD * 4 + 4 * 16 * 2 * 4;
    static constexpr int kMainBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kBytes = kMainBytes + 2 * kStages * 8 + 1024;  // + barriers + align slack
};

template <bool BF16, int HD>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const Params P,
                                                                const __grid_constant__ CUtensorMap tmK,
                                                                const __grid_constant__ CUtensorMap tmV) {
    using S = DecSmem<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kMainBytes);
    __shared__ int abort_flag;
    const uint32_t ring = smem_u32(smem);
    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = P.G * P.Tq;  // query rows per KV head (Tq = Lq here)
    const int nrc = (R + 15) / 16;
    int y = blockIdx.y;
    const int rc = y % nrc;
    y /= nrc;
    const int kvh = y % P.Hkv;
    const int b = y / P.Hkv;
    const int split = blockIdx.x;

    // This sequence's cache length: Tk, or its device-resident valid length (the
    // query block then sits at positions len - Lq .. len - 1 and keys from len on
    // are not visible), so a captured launch serves whatever lengths the buffer holds.
    int tk_b = P.Tk, qoff = P.q_offset;
    if (P.lengths) {
        tk_b = min(max(P.lengths[b], 0), P.Tk);
        qoff = tk_b - P.Tq;
    }
    // keys this CTA reads: its chunk, cut to what any of its rows can see
    int lo, hi;
    key_range(P.wl, P.wr, tk_b, qoff, qoff + P.Tq - 1, &lo, &hi);
    const int c0 = split * P.chunk, c1 = min(tk_b, c0 + P.chunk);
    lo = max(lo, c0);
    hi = min(hi, c1);
    const int t0 = lo / kKeys;
    const int ntiles = hi > lo ? (hi + kKeys - 1) / kKeys - t0 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 4);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 4) {
        // ------------------------------------------------ producer (one lane)
        if (lane == 0 && ntiles > 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            const uint64_t pol = policy_evict_first();  // streamed once
            int issued = 0;
            for (int n = 0; n < ntiles; ++n) {
                const int s = n % kStages, use = n / kStages;
                if (use > 0 && !mbar_wait(empty_bar(s), (use - 1) & 1, P.status, ST_DEC_WAIT, &abort_flag))
                    break;
                mbar_expect_tx(full_bar(s), 2 * S::kTileBytes);
                const uint32_t kdst = ring + (uint32_t)(s * 2 * S::kTileBytes);
                const uint32_t vdst = kdst + S::kTileBytes;
                const int j0 = (t0 + n) * kKeys;
#pragma unroll
                for (int bx = 0; bx < S::kBoxes; ++bx) {
                    tma_load_3d_hint(kdst + bx * kKeys * 128, &tmK, full_bar(s), kvh * HD + bx * 64, j0, b, pol);
                    tma_load_3d_hint(vdst + bx * kKeys * 128, &tmV, full_bar(s), kvh * HD + bx * 64, j0, b, pol);
                }
                issued = n + 1;
            }
            // drain: the last use of every stage must have landed before the CTA exits
            for (int n = max(0, issued - kStages); n < issued; ++n)
                mbar_wait(full_bar(n % kStages), (n / kStages) & 1, P.status, ST_DEC_WAIT | ST_TEARDOWN, nullptr);
        }
    } else {
        // --------------------------------------------------- consumers 0..3
        const int g = lane >> 2, t = lane & 3;
        int pos[2];
        bool rok[2];
        const __align__(4) uint16_t* qp[2];
        int hq[2], lqq[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int rr = rc * 16 + g + 8 * r;
            rok[r] = rr < R;
            const int gg = rok[r] ? rr / P.Tq : 0, lq = rok[r] ? rr % P.Tq : 0;
            hq[r] = kvh * P.G + gg;
            lqq[r] = lq;
            pos[r] = qoff + lq;
            qp[r] = reinterpret_cast<const uint16_t*>(P.q) + ((long long)b * P.Tq + lq) * (long long)P.H * HD +
                    (long long)hq[r] * HD;
        }
        // each row's visible keys [vlo, vhi) before the key mask (the window around its position)
        int vlo[2], vhi[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            vlo[r] = P.wl >= 0 ? max(0, pos[r] - P.wl) : 0;
            vhi[r] = P.wr >= 0 ? min(tk_b, pos[r] + P.wr + 1) : tk_b;
            if (!rok[r]) vhi[r] = vlo[r];
        }
        const float* mrow = P.key_mask ? P.key_mask + (long long)b * P.mask_bstride : nullptr;
        uint32_t qa[HD / 16][4];
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
            const int c = ks * 16 + 2 * t;
            qa[ks][0] = rok[0] ? *reinterpret_cast<const uint32_t*>(qp[0] + c) : 0u;
            qa[ks][1] = rok[1] ? *reinterpret_cast<const uint32_t*>(qp[1] + c) : 0u;
            qa[ks][2] = rok[0] ? *reinterpret_cast<const uint32_t*>(qp[0] + c + 8) : 0u;
            qa[ks][3] = rok[1] ? *reinterpret_cast<const uint32_t*>(qp[1] + c + 8) : 0u;
        }
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float o[HD / 8][4];
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        const float sl2 = P.scale_log2;
        const int kb = warp * 16;
        // ldmatrix lane roles
        const int mi = lane >> 3, ri = lane & 7;
        bool ok = true;
        for (int n = 0; n < ntiles; ++n) {
            const int s = n % kStages;
            if (!mbar_wait(full_bar(s), (n / kStages) & 1, P.status, ST_DEC_WAIT, &abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t kt = ring + (uint32_t)(s * 2 * S::kTileBytes);
            const uint32_t vt = kt + S::kTileBytes;
            const int j0 = (t0 + n) * kKeys;
            float sc[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
                // matrices: (keys kb..+7 | kb+8..+15) x (cols ks*16 | ks*16+8)
                const int key = kb + (mi >> 1) * 8 + ri;
                const int c = ks * 2 + (mi & 1);
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kt + (c >> 3) * (kKeys * 128) + sw128(key, c & 7), b00, b01, b10, b11);
                mma16816<BF16>(sc[0], qa[ks], b00, b01);
                mma16816<BF16>(sc[1], qa[ks], b10, b11);
            }
            // scale, softcap, mask -> log2 units
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = e >> 1;
                    const int j = j0 + kb + nt * 8 + 2 * t + (e & 1);
                    float x = sc[nt][e] * P.scale;
                    if (P.softcap > 0.f) x = P.softcap * tanh_accurate(x / P.softcap);
                    const bool vis = j >= vlo[r] && j < vhi[r] && (!mrow || mrow[j] > 0.5f);
                    x = vis ? x * kLog2e : -INFINITY;
                    sc[nt][e] = x;
                    mx[r] = fmaxf(mx[r], x);
                }
            (void)sl2;
            float alpha[2], ms[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mn = fmaxf(m[r], mx[r]);
                alpha[r] = mn == -INFINITY ? 1.f : fast_exp2(m[r] - mn);
                ms[r] = mn == -INFINITY ? 0.f : mn;
                m[r] = mn;
            }
            float ps[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = e >> 1;
                    const float pv = fast_exp2(sc[nt][e] - ms[r]);
                    sc[nt][e] = pv;
                    ps[r] += pv;
                }
            l[0] = l[0] * alpha[0] + ps[0];
            l[1] = l[1] * alpha[1] + ps[1];
#pragma unroll
            for (int i = 0; i < HD / 8; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[0];
                o[i][2] *= alpha[1];
                o[i][3] *= alpha[1];
            }
            uint32_t pa[4];
            pa[0] = pack2<BF16>(sc[0][0], sc[0][1]);
            pa[1] = pack2<BF16>(sc[0][2], sc[0][3]);
            pa[2] = pack2<BF16>(sc[1][0], sc[1][1]);
            pa[3] = pack2<BF16>(sc[1][2], sc[1][3]);
#pragma unroll
            for (int np = 0; np < HD / 16; ++np) {
                // matrices: (keys kb..+7 | kb+8..+15) x (cols np*16 | np*16+8), transposed
                const int key = kb + (mi & 1) * 8 + ri;
                const int c = np * 2 + (mi >> 1);
                uint32_t b0a, b1a, b0b, b1b;
                ldsm_x4_t(vt + (c >> 3) * (kKeys * 128) + sw128(key, c & 7), b0a, b1a, b0b, b1b);
                mma16816<BF16>(o[2 * np], pa, b0a, b1a);
                mma16816<BF16>(o[2 * np + 1], pa, b0b, b1b);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
        }
        // merge the four warps through shared memory (the ring is idle now)
        named_bar_sync(1, 128);
        if (ok && !abort_flag) {
            float* os = reinterpret_cast<float*>(smem);           // [4][16][HD]
            float* mls = os + 4 * 16 * HD;                        // [4][16][2]
#pragma unroll
            for (int i = 0; i < HD / 8; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = g + 8 * (e >> 1), col = i * 8 + 2 * t + (e & 1);
                    os[(warp * 16 + row) * HD + col] = o[i][e];
                }
            if (t == 0) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mls[(warp * 16 + g + 8 * r) * 2 + 0] = m[r];
                    mls[(warp * 16 + g + 8 * r) * 2 + 1] = l[r];
                }
            }
        }
        named_bar_sync(1, 128);
        if (ok && !abort_flag) {
            const float* os = reinterpret_cast<const float*>(smem);
            const float* mls = os + 4 * 16 * HD;
            for (int idx = threadIdx.x; idx < 16 * (HD + 2); idx += 128) {
                const int row = idx / (HD + 2), col = idx % (HD + 2);
                const int rr = rc * 16 + row;
                if (rr >= R) continue;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < 4; ++w) M = fmaxf(M, mls[(w * 16 + row) * 2]);
                float val = 0.f;
                if (col < HD) {
                    if (M != -INFINITY)
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const float mw = mls[(w * 16 + row) * 2];
                            if (mw != -INFINITY) val += fast_exp2(mw - M) * os[(w * 16 + row) * HD + col];
                        }
                } else if (col == HD) {
                    val = M;
                } else {
                    if (M != -INFINITY)
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const float mw = mls[(w * 16 + row) * 2];
                            if (mw != -INFINITY) val += fast_exp2(mw - M) * mls[(w * 16 + row) * 2 + 1];
                        }
                }
                const int gg = rr / P.Tq, lq = rr % P.Tq;
                const long long rowid = ((long long)b * P.H + kvh * P.G + gg) * P.Tq + lq;
                P.ws[(rowid * P.splits + split) * (HD + 2) + col] = val;
            }
        }
    }
}

// One CTA (HD threads) per query row: merge the split partials.
template <typename T, int HD>
__global__ void __launch_bounds__(HD) decode_combine_kernel(const Params P) {
    const long long rowid = blockIdx.x;  // ((b*H + h)*Lq + lq)
    const int lq = (int)(rowid % P.Tq);
    const long long bh = rowid / P.Tq;
    const int h = (int)(bh % P.H), b = (int)(bh / P.H);
    const float* rec = P.ws + rowid * P.splits * (HD + 2);
    const int d = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < P.splits; ++s) M = fmaxf(M, rec[s * (HD + 2) + HD]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < P.splits; ++s) {
            const float ms = rec[s * (HD + 2) + HD];
            if (ms == -INFINITY) continue;
            const float w = fast_exp2(ms - M);
            L += w * rec[s * (HD + 2) + HD + 1];
            acc += w * rec[s * (HD + 2) + d];
        }
    }
    T* o = reinterpret_cast<T*>(P.o) + ((long long)b * P.Tq + lq) * (long long)P.H * HD + (long long)h * HD;
    o[d] = Elem<T>::from_f(L > 0.f ? acc / L : 0.f);
    if (P.lse && d == 0) P.lse[bh * P.Tq + lq] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

template <bool BF16, int HD>
cudaError_t decode_typed(const Params& p, const DecMaps& maps, cudaStream_t s) {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const int R = p.G * p.Tq;
    const int nrc = (R + 15) / 16;
    auto k1 = decode_split_kernel<BF16, HD>;
    const int smem = DecSmem<HD>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.splits, p.B * p.Hkv * nrc);
    k1<<<grid, kThreads, smem, s>>>(p, maps.k, maps.v);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    decode_combine_kernel<T, HD><<<p.B * p.H * p.Tq, HD, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

// ----------------------------------------------- scratch for the no-alloc call
// attn_decode_noalloc keeps its split partials here instead of in a caller
// workspace, for callers that cannot allocate device memory.  Every GPU that
// loads the library holds these 32 MiB until the process exits.  Host code
// must not pass the symbol itself to a kernel: on the host it names a
// stand-in, not device memory, so the device address is looked up below.
static __device__ __align__(256) float g_decode_scratch[kDecodeScratchBytes / sizeof(float)];

cudaError_t decode_noalloc_scratch(float** out) {
    constexpr int kMaxDevices = 64;
    static float* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        // first use on this device, with it current: resolve the array's device address
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<float*>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_decode(const Params& p, int dt, const DecMaps& maps, cudaStream_t s) {
    const bool bf16 = dt == 2;
    if (p.hd == 64) return bf16 ? decode_typed<true, 64>(p, maps, s) : decode_typed<false, 64>(p, maps, s);
    if (p.hd == 256) return bf16 ? decode_typed<true, 256>(p, maps, s) : decode_typed<false, 256>(p, maps, s);
    return bf16 ? decode_typed<true, 128>(p, maps, s) : decode_typed<false, 128>(p, maps, s);
}

}  // namespace attn
