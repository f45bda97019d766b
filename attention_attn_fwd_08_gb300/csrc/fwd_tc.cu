// fwd_tc.cu -- prefill forward on the 5th-generation tensor cores (sm_103a).
//
// Computes O = softmax(st) V and LSE for fp16/bf16 inputs with fp32
// accumulation, hd 64 or 128, with causal / sliding-window / key-mask
// visibility, softcap, GQA and a query offset.
// Sources: vision_rs flash_attn2.rs, Forward (online-softmax recurrence,
// logsumexp saved for the backward); brotensor ops/flash_attention.h,
// flash_attention_decode (softcap before masking; window keys
// [p-window+1, p]) and flash_attention_forward (key mask > 0.5 keeps a key,
// fully masked key tiles are skipped); ferrotensor engine/attention.rs,
// flash_attention_v2_with (128 query rows per workgroup, GQA).
//
// One kernel, fwd_tc2_kernel: two 128-row query tiles of one (b, h) per CTA
// share every K/V tile; two softmax warpgroups alternate with the tensor core
// (details at the kernel).  Key tiles outside every row's visible range are
// never loaded; tiles that every row sees entirely skip the per-element mask.
#include <math.h>

#include <type_traits>

#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;      // query rows per tile (two tiles per CTA)
constexpr int BN = 128;      // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only when the max grows by > 256x

struct TileInfo {
    int t0, ntiles;
};

__device__ __forceinline__ TileInfo tile_range(const Params& P, int i0) {
    const int p0 = i0 + P.q_offset;
    const int p1 = min(i0 + BM, P.Tq) - 1 + P.q_offset;
    int lo, hi;
    key_range(P.causal, P.window, P.Tk, p0, p1, &lo, &hi);
    TileInfo t;
    t.t0 = lo / BN;
    t.ntiles = hi > lo ? (hi + BN - 1) / BN - t.t0 : 0;
    return t;
}

// ------------------------------------------------------------------------
// Two query tiles per CTA (256 rows of one head) sharing every K/V tile, with
// one softmax warpgroup per tile, so the tensor core works on one tile's
// P.V and next S while the other warpgroup runs its softmax (ping-pong).
//   warps 0-3  softmax of tile A (rows i0 .. i0+127)
//   warps 4-7  softmax of tile B (rows i0+128 .. i0+255)
//   warp 8     TMA producer     warp 9  TMEM owner + MMA issuer of tile A
//   warp 10    MMA issuer of tile B                                 (11 idle)
// Registers: launched at 168 per thread (384 threads = 64512); the producer
// warpgroup gives its share to the softmax warpgroups with setmaxnreg
// (2*128*224 + 128*56 = 64512, never more than the launch total).
// TMEM: S_A 0, S_B 128, O_A 256, O_B 256+hd (512 columns).  Each tile has a
// single S buffer; S_u(n) is issued after P_u(n-1) V(n-1), so a completed
// S_u(n) also means O_u is stable for a rescale.
constexpr int kThreads2 = 384;
constexpr int kRegsSoftmax = 224, kRegsProducer = 56;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsProducer <= kThreads2 * 168, "register split exceeds launch");

template <int HD>
struct Fwd2Cfg {
    static constexpr int kBoxes = HD / 64;
    static constexpr int kStages = HD == 128 ? 2 : 3;
    static constexpr int kQBytes = BM * HD * 2;
    static constexpr int kKVBytes = BN * HD * 2;
    static constexpr int kQOff = 0;  // Q_A, Q_B
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + kStages * kKVBytes;
    static constexpr int kBarOff = kVOff + kStages * kKVBytes;
    static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 2 + 1;
    static constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
    static constexpr int kLaunchBytes = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

template <bool BF16, int HD>
__global__ void __launch_bounds__(kThreads2, 1)
    fwd_tc2_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
    using C = Fwd2Cfg<HD>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    __shared__ int abort_flag;
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int Q_FULL = 0;
    auto K_FULL = [&](int s) { return 1 + s; };
    auto K_EMPTY = [&](int s) { return 1 + NS + s; };
    auto V_FULL = [&](int s) { return 1 + 2 * NS + s; };
    auto V_EMPTY = [&](int s) { return 1 + 3 * NS + s; };
    auto S_FULL = [&](int u) { return 1 + 4 * NS + u; };
    auto P_FULL = [&](int u) { return 3 + 4 * NS + u; };
    auto O_DONE = [&](int u) { return 5 + 4 * NS + u; };
    const int MMA_DONE = 7 + 4 * NS;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1-D grid, longest first: every head's last (causally heaviest) query block
    // comes before any head's next one
    const int ncta = (P.Tq + 2 * BM - 1) / (2 * BM);
    const int hb = (int)(blockIdx.x % (unsigned)(P.H * P.B));
    const int cq = ncta - 1 - (int)(blockIdx.x / (unsigned)(P.H * P.B));
    const int h = hb % P.H, b = hb / P.H, kvh = h / P.G;
    const int i0 = cq * 2 * BM;
    const bool hasB = i0 + BM < P.Tq;
    TileInfo tu[2];
    tu[0] = tile_range(P, i0);
    tu[1] = hasB ? tile_range(P, i0 + BM) : TileInfo{0, 0};
    int t0 = tu[0].t0, t1 = tu[0].t0 + tu[0].ntiles;
    if (tu[1].ntiles > 0) {
        if (tu[0].ntiles == 0) {
            t0 = tu[1].t0;
            t1 = tu[1].t0 + tu[1].ntiles;
        } else {
            t0 = min(t0, tu[1].t0);
            t1 = max(t1, tu[1].t0 + tu[1].ntiles);
        }
    }
    const int ntiles = t1 > t0 ? t1 - t0 : 0;
    auto has = [&](int u, int n) { return n >= tu[u].t0 && n < tu[u].t0 + tu[u].ntiles; };

    if (threadIdx.x == 0) {
        // stage releases and the teardown barrier take one arrival per MMA issuer
        const uint32_t issuers = hasB ? 2u : 1u;
        for (int i = 0; i < C::kNumBars; ++i) {
            uint32_t count = 1;
            if (i == P_FULL(0) || i == P_FULL(1)) count = 4;
            for (int s2 = 0; s2 < NS; ++s2)
                if (i == K_EMPTY(s2) || i == V_EMPTY(s2)) count = issuers;
            if (i == MMA_DONE) count = issuers;
            mbar_init(BAR(i), count);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (warp >= 8) {
        regs_dec<kRegsProducer>();
        if (warp == 8) {
        if (lane == 0 && ntiles > 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            const int nq = hasB ? 2 : 1;
            mbar_expect_tx(BAR(Q_FULL), nq * C::kQBytes);
            for (int u = 0; u < nq; ++u)
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    tma_load_3d(sbase + C::kQOff + u * C::kQBytes + bx * (BM * 128), &tmQ, BAR(Q_FULL),
                                h * HD + bx * 64, i0 + u * BM, b);
            int issued_k = 0, issued_v = 0;
            for (int n = 0; n < ntiles; ++n) {
                const int s = n % NS, use = n / NS;
                const int j0 = (t0 + n) * BN;
                if (use > 0 && !mbar_wait(BAR(K_EMPTY(s)), (use - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag))
                    break;
                mbar_expect_tx(BAR(K_FULL(s)), C::kKVBytes);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    tma_load_3d(sbase + C::kKOff + s * C::kKVBytes + bx * (BN * 128), &tmK, BAR(K_FULL(s)),
                                kvh * HD + bx * 64, j0, b);
                issued_k = n + 1;
                if (use > 0 && !mbar_wait(BAR(V_EMPTY(s)), (use - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag))
                    break;
                mbar_expect_tx(BAR(V_FULL(s)), C::kKVBytes);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    tma_load_3d(sbase + C::kVOff + s * C::kKVBytes + bx * (BN * 128), &tmV, BAR(V_FULL(s)),
                                kvh * HD + bx * 64, j0, b);
                issued_v = n + 1;
            }
            mbar_wait(BAR(Q_FULL), 0, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, issued_k - NS); n < issued_k; ++n)
                mbar_wait(BAR(K_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, issued_v - NS); n < issued_v; ++n)
                mbar_wait(BAR(V_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
        }
        } else if (warp == 9 || warp == 10) {
        // Two MMA issuers, one per query tile (warp 9: A, warp 10: B), so that one
        // tile's barrier waits overlap the other tile's MMA issue.  Each runs its own
        // in-order chain; both commit the K/V stage releases of every tile in the
        // union range (those barriers count one arrival per issuer).
        const int u = warp - 9;
        if (lane == 0 && ntiles > 0 && (u == 0 || hasB)) {
            constexpr uint32_t idS = idesc_f16(BF16, BM, BN, false, false);
            constexpr uint32_t idPV = idesc_f16(BF16, BM, HD, false, true);
            bool ok = mbar_wait(BAR(Q_FULL), 0, P.status, ST_FWD_MMA, &abort_flag);
            const uint64_t qdesc = sdesc_sw128(sbase + C::kQOff + u * C::kQBytes, 16, 1024);
            const uint32_t tS = tbase + u * 128, tO = tbase + 256 + u * HD;
            // n is relative to t0 here
            auto issue_s = [&](int n) -> bool {
                const int ks = n % NS;
                if (!mbar_wait(BAR(K_FULL(ks)), (n / NS) & 1, P.status, ST_FWD_MMA, &abort_flag)) return false;
                tc_fence_after();
                // descriptor + (byte offset >> 4) moves the start address (no carry below 256 KB)
                const uint64_t kdesc = sdesc_sw128(sbase + C::kKOff + ks * C::kKVBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off_q = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
                    const uint32_t off_k = ((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4;
                    mma_ss(tS, qdesc + off_q, kdesc + off_k, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR(S_FULL(u)));
                return true;
            };
            auto issue_pv = [&](int n) -> bool {
                const int vs = n % NS;
                const int k = t0 + n - tu[u].t0;  // index of this tile in u's sequence
                if (!mbar_wait(BAR(P_FULL(u)), k & 1, P.status, ST_FWD_MMA, &abort_flag)) return false;
                if (!mbar_wait(BAR(V_FULL(vs)), (n / NS) & 1, P.status, ST_FWD_MMA, &abort_flag)) return false;
                tc_fence_after();
                const uint64_t vdesc = sdesc_sw128(sbase + C::kVOff + vs * C::kKVBytes, BN * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tO, tS + kk * 8, vdesc + ((kk * 16 * 128) >> 4), idPV, (k > 0 || kk > 0) ? 1u : 0u);
                mma_commit(BAR(O_DONE(u)));
                return true;
            };
            if (ok && has(u, t0)) ok = issue_s(0);
            if (ok) mma_commit(BAR(K_EMPTY(0)));
            for (int n = 0; ok && n < ntiles; ++n) {
                if (has(u, t0 + n)) ok = issue_pv(n);
                if (ok && n + 1 < ntiles && has(u, t0 + n + 1)) ok = issue_s(n + 1);
                if (!ok) break;
                mma_commit(BAR(V_EMPTY(n % NS)));
                if (n + 1 < ntiles) mma_commit(BAR(K_EMPTY((n + 1) % NS)));
            }
            mma_commit(BAR(MMA_DONE));
            mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
        }
        }  // warps 10 and 11 only fill the producer warpgroup
    } else {
        regs_inc<kRegsSoftmax>();
        // -------------------------------------- softmax + epilogue of tile u
        const int u = warp >> 2, wq = warp & 3;
        const int r = wq * 32 + lane;
        const int ib = i0 + u * BM;  // first row of this tile
        const int i = ib + r;
        const int p = i + P.q_offset;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tbase + u * 128, tO = tbase + 256 + u * HD;
        const float sl2 = P.scale_log2;
        const bool cap = P.softcap > 0.f;
        const float cap_in = P.scale / fmaxf(P.softcap, 1e-30f);
        const float cap_out = P.softcap * kLog2e;
        const int prow0 = ib + P.q_offset, prow1 = min(ib + BM, P.Tq) - 1 + P.q_offset;
        const TileInfo my = tu[u];
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        auto wait_warp = [&](int bar, uint32_t parity) -> bool {
            const bool rr = mbar_wait(BAR(bar), parity, P.status, ST_FWD_SOFTMAX, &abort_flag);
            return __all_sync(0xffffffffu, rr);
        };
        for (int k = 0; k < my.ntiles; ++k) {
            const int j0 = (my.t0 + k) * BN;
            const bool full = tile_full(P.causal, P.window, P.Tk, prow0, prow1, j0, j0 + BN) && !P.key_mask;
            uint32_t mbits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
            if (P.key_mask) {
                const float* mrow = P.key_mask + (long long)b * P.mask_bstride;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = j0 + c * 32 + lane;
                    mbits[c] = __ballot_sync(0xffffffffu, j < P.Tk && mrow[j] > 0.5f);
                }
            }
            int clo = 0, chi = BN;
            if (!full) {
                chi = min(chi, P.Tk - j0);
                if (P.causal) chi = min(chi, p - j0 + 1);
                if (P.window > 0) {
                    clo = max(clo, p - P.window + 1 - j0);
                    if (!P.causal) chi = min(chi, p + P.window - j0);
                }
            }
            if (!wait_warp(S_FULL(u), k & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // Visibility is evaluated only in tiles that some row does not see whole
            // (kMask); s*scale and softcap*tanh(s*scale/softcap) both increase with s,
            // so row maxima are taken over raw scores and transformed once.
            auto vis_col = [&](int c) -> bool {
                return c >= clo && c < chi && ((mbits[c >> 5] >> (c & 31)) & 1u);
            };
            auto to_log2 = [&](auto capc, float raw) -> float {
                if constexpr (decltype(capc)::value) return cap_out * tanh_accurate(raw * cap_in);
                else return raw * sl2;
            };
            // raw-score row max of the tile (first tile a row sees)
            auto max_pass = [&](auto capc, auto maskc) -> float {
                constexpr bool kMask = decltype(maskc)::value;
                float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c2 = 0; c2 < 4; c2 += 2) {
                    uint32_t ta[32], tb[32];
                    tmem_ld32(tS + lane_off + c2 * 32, ta);
                    tmem_ld32(tS + lane_off + (c2 + 1) * 32, tb);
                    tmem_ld_wait_only();
                    tmem_pin(ta);
                    tmem_pin(tb);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float a = __uint_as_float(ta[e]), bb = __uint_as_float(tb[e]);
                        if constexpr (kMask) {
                            a = vis_col(c2 * 32 + e) ? a : -INFINITY;
                            bb = vis_col(c2 * 32 + 32 + e) ? bb : -INFINITY;
                        }
                        mr[e & 3] = fmaxf(mr[e & 3], fmaxf(a, bb));
                    }
                }
                const float mraw = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
                return mraw == -INFINITY ? -INFINITY : to_log2(capc, mraw);
            };
            // P = exp2(x - ms) over the tile as 16-bit pairs in registers (S stays intact in
            // TMEM until the caller stores P over it); returns the row sum and the
            // (log2-unit) row max seen along the way
            uint32_t pk[4][16];
            auto p_pass = [&](auto capc, auto maskc, float ms, float& rsum, float& mxo) {
                constexpr bool kCap = decltype(capc)::value;
                constexpr bool kMask = decltype(maskc)::value;
                float rs4[4] = {0.f, 0.f, 0.f, 0.f};
                float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                auto chunk = [&](int c, const uint32_t(&t)[32]) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float r0 = __uint_as_float(t[2 * e]), r1 = __uint_as_float(t[2 * e + 1]);
                        float x0, x1;
                        if constexpr (kCap) {
                            x0 = fmaf(cap_out, tanh_accurate(r0 * cap_in), -ms);
                            x1 = fmaf(cap_out, tanh_accurate(r1 * cap_in), -ms);
                        } else {
                            x0 = fmaf(r0, sl2, -ms);
                            x1 = fmaf(r1, sl2, -ms);
                        }
                        if constexpr (kMask) {
                            // the mask goes on the transformed argument: softcap*tanh(-inf) is finite
                            const bool v0 = vis_col(c * 32 + 2 * e), v1 = vis_col(c * 32 + 2 * e + 1);
                            r0 = v0 ? r0 : -INFINITY;
                            r1 = v1 ? r1 : -INFINITY;
                            x0 = v0 ? x0 : -INFINITY;
                            x1 = v1 ? x1 : -INFINITY;
                        }
                        mr[e & 3] = fmaxf(mr[e & 3], fmaxf(r0, r1));
                        const float p0 = fast_exp2(x0);  // masked: ex2(-inf) = 0
                        const float p1 = fast_exp2(x1);
                        rs4[e & 3] += p0 + p1;
                        pk[c][e] = pack2<BF16>(p0, p1);
                    }
                };
                uint32_t ta[32], tb[32];
                tmem_ld32(tS + lane_off + 0 * 32, ta);
                tmem_ld_wait(ta);
                tmem_ld32(tS + lane_off + 1 * 32, tb);
                chunk(0, ta);
                tmem_ld_wait(tb);
                tmem_ld32(tS + lane_off + 2 * 32, ta);
                chunk(1, tb);
                tmem_ld_wait(ta);
                tmem_ld32(tS + lane_off + 3 * 32, tb);
                chunk(2, ta);
                tmem_ld_wait(tb);
                chunk(3, tb);
                rsum = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
                const float mraw = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
                mxo = mraw == -INFINITY ? -INFINITY : to_log2(capc, mraw);
            };
            auto run_tile = [&](auto capc, auto maskc) {
                // rows that have seen no key yet take this tile's max as their reference
                if (__any_sync(0xffffffffu, l == 0.f)) {
                    const float mt = max_pass(capc, maskc);
                    if (l == 0.f) m_used = fmaxf(m_used, mt);
                }
                // one pass against the running reference max; if some row's max grew
                // by more than 2^8 (rare), rescale O, move the reference and redo the tile
                float rs, mx;
                p_pass(capc, maskc, m_used == -INFINITY ? 0.f : m_used, rs, mx);
                const bool resc = l > 0.f && mx > m_used + kRescaleThreshold;
                if (__any_sync(0xffffffffu, resc)) {
                    // S_u(k) completed after P_u(k-1) V(k-1): O_u already holds it
                    const float alpha = fast_exp2(resc ? m_used - mx : 0.f);
                    if (resc) {
                        m_used = mx;
                        l *= alpha;
                    }
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t orr[32];
                        tmem_ld32(tO + lane_off + c * 32, orr);
                        tmem_ld_wait(orr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(tO + lane_off + c * 32, orr);
                    }
                    // S is still intact in TMEM: recompute this tile's P against the new max
                    p_pass(capc, maskc, m_used == -INFINITY ? 0.f : m_used, rs, mx);
                }
                l += rs;
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_st16(tS + lane_off + c * 16, pk[c]);
            };
            using TT = std::integral_constant<bool, true>;
            using FF = std::integral_constant<bool, false>;
            if (cap) {
                if (full) run_tile(TT(), FF());
                else run_tile(TT(), TT());
            } else {
                if (full) run_tile(FF(), FF());
                else run_tile(FF(), TT());
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(P_FULL(u)));
        }
        using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
        const bool row_ok = i < P.Tq;
        T* orow = reinterpret_cast<T*>(P.o) + ((long long)b * P.Tq + (row_ok ? i : 0)) * (long long)P.H * HD +
                  (long long)h * HD;
        const bool have_o = ok && my.ntiles > 0 && wait_warp(O_DONE(u), (my.ntiles - 1) & 1);
        if (have_o) tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
            uint32_t orr[32];
            if (have_o) {
                tmem_ld32(tO + lane_off + c * 32, orr);
                tmem_ld_wait(orr);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) orr[e] = 0u;
            }
            if (row_ok && (have_o || my.ntiles == 0)) {
                uint32_t packed[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    packed[e] = pack2<BF16>(__uint_as_float(orr[2 * e]) * inv, __uint_as_float(orr[2 * e + 1]) * inv);
                uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
            }
        }
        if (row_ok && P.lse && (have_o || my.ntiles == 0))
            P.lse[((long long)b * P.H + h) * P.Tq + i] =
                l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

template <bool BF16, int HD>
cudaError_t fwd2_typed(const Params& p, const FwdMaps& m, cudaStream_t s) {
    using C = Fwd2Cfg<HD>;
    auto kern = fwd_tc2_kernel<BF16, HD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kLaunchBytes);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((p.Tq + 2 * BM - 1) / (2 * BM)) * p.H * p.B;
    kern<<<grid, kThreads2, C::kLaunchBytes, s>>>(p, m.q, m.k, m.v);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fwd(const Params& p, int dt, const FwdMaps& maps, cudaStream_t s) {
    const bool bf16 = dt == 2;
    if (p.hd == 64) return bf16 ? fwd2_typed<true, 64>(p, maps, s) : fwd2_typed<false, 64>(p, maps, s);
    return bf16 ? fwd2_typed<true, 128>(p, maps, s) : fwd2_typed<false, 128>(p, maps, s);
}

}  // namespace attn
