// fwd_hd256.cuh -- prefill forward at head size 256 on the tcgen05 tensor cores.
//
// Computes O = softmax(st) V and LSE for fp16/bf16 inputs with fp32
// accumulation at hd 256, with causal / sliding-window / key-mask visibility,
// softcap, GQA and a query offset (dense batches).
// Sources: vision_rs flash_attn2.rs, Forward (online-softmax recurrence,
// logsumexp saved for the backward); brotensor ops/flash_attention.h,
// flash_attention_decode_len (the grouped kernel serves head sizes 64, 128 and
// 256) and flash_attention_decode (softcap before masking; window keys
// [p-window+1, p]).
//
// At hd 256 one 128-row query tile fills half of TMEM with its O accumulator
// (256 columns), so a CTA works on one query tile at a time and overlaps its
// softmax with the tensor core by double-buffering S instead:
//   TMEM  S_0 0..63, S_1 64..127 (64-key score tiles), Q 128..255 (the query
//         tile as 16-bit pairs, the A operand of S = Q K^T), O 256..511.
//   The MMA warp issues S(n+1) (and S(n+2) once P(n) V(n) is issued) while the
//   softmax warps work on S(n): S(n+2) goes into S(n)'s buffer after P(n) V(n)
//   has read P(n) from it (tcgen05 MMAs of one thread run in order).  With Q in
//   TMEM both GEMMs read one operand from shared memory: K (64 B per clock at
//   N = 64) and V (N = 256).
// Warps: 0-3 softmax (one thread per query row; they also copy Q into TMEM and
// write O), 4 TMA producer (Q, then 64-key K and V tiles into a 2-stage ring,
// 128-byte swizzle), 5 TMEM owner and MMA issuer.  Persistent: one CTA per SM
// walks 128-row work items in snake order, longest first.
#pragma once

#include <math.h>

#include <type_traits>

#include "kernels.h"

namespace attn {
namespace {

namespace h256 {

constexpr int HD = 256;
constexpr int BM = 128;  // query rows per work item
constexpr int BN = 64;   // keys per tile
constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr int kBoxes = HD / 64;                 // 64-column TMA boxes per row
constexpr int kQBytes = BM * HD * 2;            // 64 KB
constexpr int kKVBytes = BN * HD * 2;           // 32 KB per K (or V) tile
constexpr int kQOff = 0;
constexpr int kKOff = kQBytes;
constexpr int kVOff = kKOff + kStages * kKVBytes;
constexpr int kBarOff = kVOff + kStages * kKVBytes;
constexpr int kNumBars = 14 + 4 * kStages;
constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
constexpr int kLaunchBytes = kBytes + 1024;
constexpr float kLog2e = 1.4426950408889634f;
// Reference band (log2 units): a tile's row max may lie up to kHi above the row's
// reference, and a row's first visible tile must put its max at kLo or above;
// 16-bit P then stays within [2^-2, 2^8] at the row max.
constexpr float kHi = 8.0f, kLo = -2.0f;

struct Item {
    int b, h, kvh, i0;
    int t0, ntiles;  // key tiles of 64 the rows see
};
__device__ __forceinline__ int num_items(const Params& P) { return (P.Tq + BM - 1) / BM * P.H * P.B; }
// item w: query block qb (longest first: every head's last block before any head's next)
__device__ __forceinline__ Item item_of(const Params& P, int w) {
    Item it;
    const int nqb = (P.Tq + BM - 1) / BM;
    const int hb = w % (P.H * P.B);
    it.h = hb % P.H;
    it.b = hb / P.H;
    it.kvh = it.h / P.G;
    it.i0 = (nqb - 1 - w / (P.H * P.B)) * BM;
    int lo, hi;
    key_range(P.wl, P.wr, P.Tk, it.i0 + P.q_offset, min(it.i0 + BM, P.Tq) - 1 + P.q_offset, &lo, &hi);
    it.t0 = lo / BN;
    it.ntiles = hi > lo ? (hi + BN - 1) / BN - it.t0 : 0;
    return it;
}

}  // namespace h256

// MODE 0: dense; MODE 4: dense with a softcap.
template <bool BF16, int MODE>
__global__ void __launch_bounds__(h256::kThreads, 1)
    fwd_hd256_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
    using namespace h256;
    constexpr bool kCap = (MODE & 4) != 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    __shared__ int abort_flag;
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int Q_FULL = 0;    // the item's Q tile in shared memory (TMA)
    const int Q_EMPTY = 1;   // ... copied out of shared memory (4 softmax warps)
    const int QT_READY = 2;  // Q of the item in TMEM (4 softmax warps)
    const int QT_EMPTY = 3;  // the item's last S completed: TMEM Q may be replaced
    const int P_FULL = 4;    // P of a tile in TMEM (4 softmax warps)
    const int PV_DONE = 5;   // a tile's P.V completed
    const int O_DONE = 6;    // the item's last P.V completed
    const int O_EMPTY = 7;   // the epilogue has read O out of TMEM (4 softmax warps)
    const int MMA_DONE = 8;
    auto S_FULL = [&](int bf) { return 9 + bf; };
    auto K_FULL = [&](int s) { return 11 + s; };
    auto K_EMPTY = [&](int s) { return 11 + kStages + s; };
    auto V_FULL = [&](int s) { return 11 + 2 * kStages + s; };
    auto V_EMPTY = [&](int s) { return 11 + 3 * kStages + s; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = num_items(P);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool four = i == Q_EMPTY || i == QT_READY || i == P_FULL || i == O_EMPTY;
            mbar_init(BAR(i), four ? 4 : 1);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tQ = tbase + 128, tO = tbase + 256;

    if (warp == 4) {
        // ---------------------------------------------- TMA producer (whole warp)
        if (elect_one()) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
        bool ok = true;
        int qn = 0, gk = 0, gv = 0;  // Q, K and V loads so far
        for (int kw = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++kw)) {
            const Item it = item_of(P, w);
            if (it.ntiles == 0) continue;
            if (qn > 0 && !warp_wait(BAR(Q_EMPTY), (qn - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag)) break;
            if (elect_one()) mbar_expect_tx(BAR(Q_FULL), kQBytes);
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
                if (elect_one())
                    tma_load_3d(sbase + kQOff + bx * (BM * 128), &tmQ, BAR(Q_FULL), it.h * HD + bx * 64, it.i0, it.b);
            ++qn;
            for (int n = 0; ok && n < it.ntiles; ++n) {
                const int s = gk % kStages, use = gk / kStages;
                const int j0 = (it.t0 + n) * BN;
                if (use > 0 && !warp_wait(BAR(K_EMPTY(s)), (use - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) mbar_expect_tx(BAR(K_FULL(s)), kKVBytes);
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx)
                    if (elect_one())
                        tma_load_3d(sbase + kKOff + s * kKVBytes + bx * (BN * 128), &tmK, BAR(K_FULL(s)),
                                    it.kvh * HD + bx * 64, j0, it.b);
                ++gk;
                if (use > 0 && !warp_wait(BAR(V_EMPTY(s)), (use - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) mbar_expect_tx(BAR(V_FULL(s)), kKVBytes);
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx)
                    if (elect_one())
                        tma_load_3d(sbase + kVOff + s * kKVBytes + bx * (BN * 128), &tmV, BAR(V_FULL(s)),
                                    it.kvh * HD + bx * 64, j0, it.b);
                ++gv;
            }
        }
        // every copy in flight lands before the CTA exits
        if (qn > 0) mbar_wait(BAR(Q_FULL), (qn - 1) & 1, P.status, ST_TEARDOWN, nullptr);
        for (int n = max(0, gk - kStages); n < gk; ++n)
            mbar_wait(BAR(K_FULL(n % kStages)), (n / kStages) & 1, P.status, ST_TEARDOWN, nullptr);
        for (int n = max(0, gv - kStages); n < gv; ++n)
            mbar_wait(BAR(V_FULL(n % kStages)), (n / kStages) & 1, P.status, ST_TEARDOWN, nullptr);
    } else if (warp == 5) {
        // ---------------------------------------------- MMA issuer (whole warp)
        constexpr uint32_t idS = idesc_f16(BF16, BM, BN, false, false);
        constexpr uint32_t idPV = idesc_f16(BF16, BM, HD, false, true);
        auto wait_all = [&](int bar, uint32_t parity) -> bool {
            return warp_wait(BAR(bar), parity, P.status, ST_FWD_MMA, &abort_flag);
        };
        bool ok = true;
        int gt = 0;   // key tiles so far (ring position and S buffer)
        int act = 0;  // items with tiles so far
        // S(t) = Q K(t)^T into buffer t & 1, A from TMEM; after the item's last S, the
        // TMEM copy of Q is free once that S completes (QT_EMPTY)
        auto issue_s = [&](int t, bool last) -> bool {
            const int s = t % kStages;
            if (!wait_all(K_FULL(s), (t / kStages) & 1)) return false;
            tc_fence_after();
            const uint64_t kdesc = sdesc_sw128(sbase + kKOff + s * kKVBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t boff = ((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4;
                mma_ts_e(tbase + (t & 1) * 64, tQ + kk * 8, kdesc + boff, idS, kk > 0 ? 1u : 0u);
            }
            mma_commit_e(BAR(S_FULL(t & 1)));
            mma_commit_e(BAR(K_EMPTY(s)));
            if (last) mma_commit_e(BAR(QT_EMPTY));
            return true;
        };
        for (int kw = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++kw)) {
            const Item it = item_of(P, w);
            if (it.ntiles == 0) continue;
            ok = wait_all(QT_READY, act & 1);
            if (ok) ok = issue_s(gt, it.ntiles == 1);
            if (ok && it.ntiles > 1) ok = issue_s(gt + 1, it.ntiles == 2);
            for (int n = 0; ok && n < it.ntiles; ++n) {
                const int t = gt + n, s = t % kStages;
                ok = wait_all(P_FULL, t & 1);
                // the first P.V overwrites O: the previous item's epilogue must have read it
                if (ok && n == 0 && act > 0) ok = wait_all(O_EMPTY, (act - 1) & 1);
                if (ok) ok = wait_all(V_FULL(s), (t / kStages) & 1);
                if (!ok) break;
                tc_fence_after();
                // O (+)= P V(t): P is 16-bit in the first 32 columns of S(t)'s buffer
                const uint64_t vdesc = sdesc_sw128(sbase + kVOff + s * kKVBytes, BN * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts_e(tO, tbase + (t & 1) * 64 + kk * 8, vdesc + ((kk * 16 * 128) >> 4), idPV,
                               (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit_e(BAR(V_EMPTY(s)));
                mma_commit_e(BAR(PV_DONE));
                if (n == it.ntiles - 1) mma_commit_e(BAR(O_DONE));
                if (n + 2 < it.ntiles) ok = issue_s(t + 2, n + 2 == it.ntiles - 1);
            }
            gt += it.ntiles;
            ++act;
        }
        mma_commit_e(BAR(MMA_DONE));
        mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
    } else if (warp < 4) {
        // ------------------------------------ softmax + epilogue, one thread per row
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sl2 = P.scale_log2;
        const uint64_t sl2_2 = f2_make(sl2, sl2);
        const float cap_in = P.scale / fmaxf(P.softcap, 1e-30f);
        const float cap_out = P.softcap * kLog2e;
        auto wait_warp = [&](int bar, uint32_t parity) -> bool {
            const bool rr = mbar_wait(BAR(bar), parity, P.status, ST_FWD_SOFTMAX, &abort_flag);
            return __all_sync(0xffffffffu, rr);
        };
        bool ok = true;
        int gt = 0, act = 0, qc = 0;  // key tiles, items with tiles and Q copies so far
        for (int kw = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++kw)) {
            const Item it = item_of(P, w);
            if (it.i0 >= P.Tq) continue;
            const int i = it.i0 + r;
            const int p = i + P.q_offset;
            const int prow0 = it.i0 + P.q_offset, prow1 = min(it.i0 + BM, P.Tq) - 1 + P.q_offset;
            float m_used = 0.f, l = 0.f;
            if (it.ntiles > 0) {
                // Q into TMEM: the previous item's S MMAs must have finished reading it
                if (qc > 0) ok = wait_warp(QT_EMPTY, (qc - 1) & 1);
                if (ok) ok = wait_warp(Q_FULL, qc & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx) {
                    uint32_t wv[32];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(smem + kQOff + bx * (BM * 128) + r * 128 +
                                                                         ((ch ^ (r & 7)) << 4));
                        wv[4 * ch] = v4.x;
                        wv[4 * ch + 1] = v4.y;
                        wv[4 * ch + 2] = v4.z;
                        wv[4 * ch + 3] = v4.w;
                    }
                    tmem_st32(tQ + lane_off + bx * 32, wv);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(BAR(Q_EMPTY));   // the shared-memory tile may be reloaded
                    mbar_arrive(BAR(QT_READY));  // the MMA warp may start this item
                }
                ++qc;
            }
            for (int n = 0; ok && n < it.ntiles; ++n) {
                const int t = gt + n, bf = t & 1;
                const uint32_t tS = tbase + bf * 64;
                const int j0 = (it.t0 + n) * BN;
                uint32_t mbits[2] = {0xffffffffu, 0xffffffffu};
                if (P.key_mask) {
                    const float* mrow = P.key_mask + (long long)it.b * P.mask_bstride;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int j = j0 + c * 32 + lane;
                        mbits[c] = __ballot_sync(0xffffffffu, j < P.Tk && mrow[j] > 0.5f);
                    }
                }
                const bool full = tile_full(P.wl, P.wr, P.Tk, prow0, prow1, j0, j0 + BN) &&
                                  (mbits[0] & mbits[1]) == 0xffffffffu;
                int clo = 0, chi = BN;
                if (!full) {
                    chi = min(chi, P.Tk - j0);
                    if (P.wr >= 0) chi = min(chi, p + P.wr - j0 + 1);
                    if (P.wl >= 0) clo = max(clo, p - P.wl - j0);
                    if (i >= P.Tq) chi = 0;
                }
                if (!wait_warp(S_FULL(bf), (t >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[2][32];
                tmem_ld32(tS + lane_off, sv[0]);
                tmem_ld32(tS + lane_off + 32, sv[1]);
                tmem_ld_wait_only();
                tmem_pin(sv[0]);
                tmem_pin(sv[1]);
                // softcap: the fitted polynomial serves the tile unless a raw score of
                // the warp's rows lies outside its range (then the exp-based tanh)
                bool poly = false;
                if constexpr (kCap) {
                    float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const int q = 2 * c + ((e >> 2) & 1);
                            am[q] = max3f(am[q], fabsf(__uint_as_float(sv[c][e])), fabsf(__uint_as_float(sv[c][e + 1])));
                            am[q] = max3f(am[q], fabsf(__uint_as_float(sv[c][e + 2])),
                                          fabsf(__uint_as_float(sv[c][e + 3])));
                        }
                    const CapPoly cp = cap_poly(P.scale, P.softcap);
                    poly = __all_sync(0xffffffffu, fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])) <= cp.r_max) &&
                           (full || cp.inf_ok);
                }
                if (!full) {
                    // invisible scores become -inf: [clo, chi) and the key mask
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int lo = min(max(clo - 32 * c, 0), 32), hi = min(max(chi - 32 * c, 0), 32);
                        const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
                        const uint32_t below_lo = lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u);
                        const uint32_t vw = below_hi & ~below_lo & mbits[c];
#pragma unroll
                        for (int e = 0; e < 32; ++e) sv[c][e] = ((vw >> e) & 1u) ? sv[c][e] : 0xff800000u;
                    }
                }
                // x of a pair of raw scores: (capped) score * log2(e) - m
                auto to_x = [&](auto modec, uint64_t rr, uint64_t nms) -> uint64_t {
                    constexpr int kMode = decltype(modec)::value;
                    if constexpr (kMode == 2) {
                        float r0, r1, m0, m1;
                        f2_split(rr, r0, r1);
                        f2_split(nms, m0, m1);
                        // a masked score is -inf, and softcap*tanh(-inf) would be finite
                        return f2_make(r0 == -INFINITY ? -INFINITY : fmaf(cap_out, tanh_accurate(r0 * cap_in), m0),
                                       r1 == -INFINITY ? -INFINITY : fmaf(cap_out, tanh_accurate(r1 * cap_in), m1));
                    } else if constexpr (kMode == 1) {
                        // x = r * (sl2 + u * S'(u)) + m with u = r^2 and S' the fit's S with
                        // scale * log2(e) folded in
                        const CapPoly cp = cap_poly(P.scale, P.softcap);
                        const uint64_t u = f2_mul(rr, rr);
                        uint64_t sp = f2_fma(u, f2_mul(cp.s3, sl2_2), f2_mul(cp.s2, sl2_2));
                        sp = f2_fma(u, sp, f2_mul(cp.s1, sl2_2));
                        sp = f2_fma(u, sp, f2_mul(cp.s0, sl2_2));
                        return f2_fma(rr, f2_fma(u, sp, sl2_2), nms);
                    } else {
                        return f2_fma(rr, sl2_2, nms);
                    }
                };
                // pass 1: row max
                float rm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int q = 2 * c + ((e >> 2) & 1);
                        rm[q] = max3f(rm[q], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
                        rm[q] = max3f(rm[q], __uint_as_float(sv[c][e + 2]), __uint_as_float(sv[c][e + 3]));
                    }
                const float rmax = fmaxf(fmaxf(rm[0], rm[1]), fmaxf(rm[2], rm[3]));
                float xm, xm_;
                {
                    const uint64_t r2 = f2_make(rmax, rmax), n2 = f2_make(-m_used, -m_used);
                    uint64_t x2;
                    if constexpr (!kCap) x2 = to_x(std::integral_constant<int, 0>(), r2, n2);
                    else x2 = to_x(std::integral_constant<int, 2>(), r2, n2);
                    f2_split(x2, xm, xm_);
                }
                if (rmax == -INFINITY) xm = -INFINITY;
                // The reference m moves only when P would leave [2^-2, 2^8] at the row max;
                // then O (which holds every earlier tile of the item once P(t-1) V(t-1)
                // completed) is rescaled in TMEM first.
                const bool resc = xm > kHi || (l == 0.f && xm < kLo && xm != -INFINITY);
                if (__any_sync(0xffffffffu, resc)) {
                    const float alpha = fast_exp2(resc && l > 0.f ? -xm : 0.f);
                    if (resc) {
                        m_used += xm;
                        l *= alpha;
                    }
                    if (n > 0) {
                        // P(t-2) V(t-2) completed before S(t) (issued after it); wait for P(t-1) V(t-1)
                        if (!wait_warp(PV_DONE, (t - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < HD / 32; ++c) {
                            uint32_t orr[32];
                            tmem_ld32(tO + lane_off + c * 32, orr);
                            tmem_ld_wait(orr);
#pragma unroll
                            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                            tmem_st32(tO + lane_off + c * 32, orr);
                        }
                    }
                }
                // pass 2: P over the first 32 columns of S's buffer, 16 at a time
                auto p_pass = [&](auto modec) {
                    const uint64_t nms = f2_make(-m_used, -m_used);
                    uint64_t rs2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float x0, x1;
                            f2_split(to_x(modec, f2_make(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])),
                                          nms),
                                     x0, x1);
                            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                            rs2[e & 1] = f2_add(rs2[e & 1], f2_make(p0, p1));
                            pk[e] = pack2<BF16>(p0, p1);
                        }
                        tmem_st16(tS + lane_off + c * 16, pk);
                    }
                    float a0, a1, b0, b1;
                    f2_split(rs2[0], a0, a1);
                    f2_split(rs2[1], b0, b1);
                    l += (a0 + b0) + (a1 + b1);
                };
                if constexpr (!kCap) p_pass(std::integral_constant<int, 0>());
                else if (poly) p_pass(std::integral_constant<int, 1>());
                else p_pass(std::integral_constant<int, 2>());
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(P_FULL));
            }
            if (!ok) break;
            // epilogue: O / l of this row, 32 columns at a time (zero when no key is seen)
            bool have_o = false;
            if (it.ntiles > 0) {
                if (!wait_warp(O_DONE, act & 1)) break;
                tc_fence_after();
                have_o = true;
                ++act;
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(P.o) +
                                                   (((long long)it.b * P.Tq + i) * P.H + it.h) * HD);
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t orr[32];
                if (have_o) {
                    tmem_ld32(tO + lane_off + c * 32, orr);
                    tmem_ld_wait(orr);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) orr[e] = 0u;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack2<BF16>(__uint_as_float(orr[2 * e]) * inv, __uint_as_float(orr[2 * e + 1]) * inv);
                if (i < P.Tq) {
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4)
                        orow[c * 4 + w4] = make_uint4(pk[4 * w4], pk[4 * w4 + 1], pk[4 * w4 + 2], pk[4 * w4 + 3]);
                }
            }
            // O is in registers and stored: the next item's first P.V may overwrite it
            if (have_o) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(O_EMPTY));
            }
            if (P.lse && i < P.Tq)
                P.lse[((long long)it.b * P.H + it.h) * P.Tq + i] =
                    l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
            gt += it.ntiles;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

template <bool BF16>
cudaError_t fwd_hd256_typed(const Params& p, const FwdMaps& m, cudaStream_t s) {
    auto kern = p.softcap > 0.f ? fwd_hd256_kernel<BF16, 4> : fwd_hd256_kernel<BF16, 0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, h256::kLaunchBytes);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long items = (long long)((p.Tq + h256::BM - 1) / h256::BM) * p.H * p.B;
    const unsigned grid = (unsigned)(items < nsm ? items : nsm);
    kern<<<grid, h256::kThreads, h256::kLaunchBytes, s>>>(p, m.q, m.k, m.v);
    return cudaGetLastError();
}

}  // namespace

}  // namespace attn
