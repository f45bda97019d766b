// bwd_hd256.cuh -- backward at head size 256 on the tcgen05 tensor cores.
//
// Computes dQ, dK, dV of O = softmax(st) V for fp16/bf16 inputs with fp32
// accumulation at hd 256 (dense batches: causal / sliding-window / key-mask
// visibility, softcap, GQA, query offset), recomputing P = exp(st - LSE) from the
// saved LSE.  D = rowsum(dO*O) and -LSE*log2(e) come from the preprocess pass in
// the workspace.
// Sources: vision_rs flash_attn2.rs, "Backward - dQ" and "Backward - dK / dV"
// (p = exp(s*scale - L), dS = p (dO.V - D), dQ += dS K scale, dK += dS Q scale,
// dV += p dO); forge attention.metal, attention_bwd_dq_f32 / attention_bwd_dkv_f32
// (softcap derivative 1 - tanh^2 of the uncapped score, dK/dV summed over the query
// heads sharing a KV head, no atomics); brotensor ops/flash_attention.h,
// flash_attention_decode_len (the grouped kernel serves head sizes 64, 128 and 256).
//
// At hd 256 a 128-row accumulator takes 256 TMEM columns, so dK and dV of a key
// block cannot share one SM's 512: they come from two launches of one kernel, each
// recomputing S^T.
//   dV pass (PART 1): TMEM S^T 0 / 64 (double buffer; P^T as 16-bit pairs over the
//     first 32 columns), dV 256..511.  MMAs: S^T = K Q^T (SS), dV += P^T dO (TS).
//   dK pass (PART 2): TMEM S^T 0..63, dP^T 64..127, V 128..255 (16-bit pairs, the A
//     operand of dP^T = V dO^T), dK 256..511.  MMAs: S^T (SS), dP^T (TS), dK += dS^T Q
//     (TS, dS^T over the first 32 columns of S^T).  S^T and dP^T are single-buffered.
//   CTA = 128 keys of one (b, kv head): warps 0-3 one key row per thread, 4 TMA
//   producer (K once, then 64-row Q and dO tiles of every query head of the group into
//   two two-stage rings), 5 TMEM owner and MMA issuer.  The ring that the tile's first
//   MMAs alone read (Q in the dV pass, dO in the dK pass) is released as soon as they
//   complete, so its next load runs under the rest of the tile; the other ring carries
//   the tile's -LSE*log2(e) and -D and is released by the accumulating MMA.
// dQ pass: CTA = 128 query rows of one (b, h) over 64-key tiles.  TMEM S 0..63, dP
//   64..127 (single-buffered), Q 128..255 (16-bit pairs, the A operand of S = Q K^T),
//   dQ 256..511.  MMAs: S (TS), dP = dO V^T (SS), dQ += dS K (TS, dS over S).  dO stays
//   in shared memory; Q passes through the first ring stage on its way into TMEM.
#pragma once

#include <math.h>

#include <type_traits>

#include "kernels.h"

namespace attn {
namespace {

namespace b256 {

constexpr int HD = 256;
constexpr int kBoxes = HD / 64;  // 64-column TMA boxes per row
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 192;    // 4 compute warps, producer, MMA issuer

// ------------------------------------------------------------- dK / dV passes
constexpr int BKV = 128;                   // keys per CTA
constexpr int BQ = 64;                     // query rows per tile
constexpr int kKBytes = BKV * HD * 2;      // 64 KB: the key block's K (V passes through the ring)
constexpr int kTBytes = BQ * HD * 2;       // 32 KB: one Q or dO tile
constexpr int kKVStages = 2;
constexpr int kKOff = 0;
constexpr int kRingOff = kKBytes;          // the Q ring (stage s at + s * kTBytes), then the dO ring
constexpr int kGRingOff = kRingOff + kKVStages * kTBytes;
constexpr int kStatOff = kGRingOff + kKVStages * kTBytes;  // [stage][2][BQ] floats: -LSE*log2e, -D
constexpr int kStatBytes = 2 * BQ * 4;
constexpr int kKVBarOff = kStatOff + kKVStages * kStatBytes;
constexpr int kKVNumBars = 18;
constexpr int kKVLaunchBytes = kKVBarOff + kKVNumBars * 8 + 16 + 1024;
static_assert(kKVLaunchBytes <= 227 * 1024, "shared memory");

// ------------------------------------------------------------------ dQ pass
constexpr int BQD = 128;                   // query rows per CTA
constexpr int BKD = 64;                    // keys per tile
constexpr int kDoBytes = BQD * HD * 2;     // 64 KB
constexpr int kKTileBytes = BKD * HD * 2;  // 32 KB per K (or V) tile
constexpr int kDqStages = 2;
constexpr int kDoOff = 0;
constexpr int kDqRingOff = kDoBytes;       // stage s: K, then V (stage 0 first holds Q)
constexpr int kDqBarOff = kDqRingOff + kDqStages * 2 * kKTileBytes;
constexpr int kDqNumBars = 16;
constexpr int kDqLaunchBytes = kDqBarOff + kDqNumBars * 8 + 16 + 1024;
static_assert(kDqLaunchBytes <= 227 * 1024, "shared memory");
static_assert(BQD * HD * 2 == 2 * kKTileBytes, "Q passes through one ring stage");

}  // namespace b256

// The additive-free score transform of both passes: x = (capped) score * log2(e) +
// nl (nl = -LSE*log2(e)), P = 2^x, and the softcap's derivative 1 - tanh^2 of the
// uncapped score (1 without a softcap).  A masked score is -inf and gives P = 0.
template <bool CAP>
__device__ __forceinline__ float b256_p(const Params& P, float s, float nl, float& dcap) {
    if constexpr (!CAP) {
        dcap = 1.f;
        return fast_exp2(fmaf(s, P.scale_log2, nl));
    } else {
        if (s == -INFINITY) {
            dcap = 0.f;
            return 0.f;
        }
        const float t = tanh_accurate(s * (P.scale / P.softcap));
        dcap = fmaf(-t, t, 1.f);
        return fast_exp2(fmaf(P.softcap * b256::kLog2e, t, nl));
    }
}

// PART 1: dV of a 128-key block; PART 2: dK.  MODE 0: dense; MODE 4: with a softcap.
template <bool BF16, int MODE, int PART>
__global__ void __launch_bounds__(b256::kThreads, 1)
    bwd_h256_kv_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG) {
    using namespace b256;
    constexpr bool kCap = (MODE & 4) != 0, kDK = PART == 2;
    constexpr int NS = kKVStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kKVBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kKVNumBars);
    const float* stat = reinterpret_cast<const float*>(smem + kStatOff);
    __shared__ int abort_flag;
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int K_FULL = 0;
    const int V_FULL = 1;     // (dK pass) V of the key block in the Q ring's space
    const int V_COPIED = 2;   // ... copied into TMEM (4 compute warps)
    const int ACC_DONE = 3;
    const int MMA_DONE = 4;
    auto Q_FULL = [&](int s) { return 5 + s; };
    auto Q_EMPTY = [&](int s) { return 7 + s; };
    auto G_FULL = [&](int s) { return 9 + s; };      // dO
    auto G_EMPTY = [&](int s) { return 11 + s; };
    auto ST_FULL = [&](int bf) { return 13 + bf; };  // S^T (and dP^T) of a tile in TMEM
    auto PT_FULL = [&](int bf) { return 15 + bf; };  // P^T (dS^T) of a tile in TMEM (4 compute warps)
    // the ring that carries the statistics and is released by the accumulating MMA
    auto L_FULL = [&](int s) { return kDK ? Q_FULL(s) : G_FULL(s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // key blocks in order, every (b, kv head)'s block kb before any one's block kb + 1
    // (causally the first are seen by the most queries: the heaviest CTAs start first)
    const int ng = P.Hkv * P.B;
    const int kb = (int)blockIdx.x / ng, kg = (int)blockIdx.x % ng;
    const int kvh = kg % P.Hkv, b = kg / P.Hkv;
    const int j0 = kb * BKV;
    int qlo, qhi;
    query_range(P.wl, P.wr, P.Tq, P.q_offset, j0, min(j0 + BKV, P.Tk), &qlo, &qhi);
    const int qt0 = qlo / BQ;
    const int nqt = qhi > qlo ? (qhi + BQ - 1) / BQ - qt0 : 0;
    const int ntiles = nqt * P.G;  // (head, query tile) pairs, head-major
    auto tile_head = [&](int n) { return kvh * P.G + n / max(nqt, 1); };
    auto tile_i0 = [&](int n) { return (qt0 + n % max(nqt, 1)) * BQ; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kKVNumBars; ++i)
            mbar_init(BAR(i), (i == V_COPIED || i == PT_FULL(0) || i == PT_FULL(1)) ? 4 : 1);
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
    const uint32_t tAcc = tbase + 256, tV = tbase + 128;

    if (warp == 4) {
        // ---------------------------------------------- TMA producer (whole warp)
        if (ntiles > 0) {
            if (elect_one()) {
                prefetch_tmap(&tmQ);
                prefetch_tmap(&tmK);
                prefetch_tmap(&tmG);
                if (kDK) prefetch_tmap(&tmV);
            }
            if (elect_one()) mbar_expect_tx(BAR(K_FULL), kKBytes);
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
                if (elect_one())
                    tma_load_3d(sbase + kKOff + bx * (BKV * 128), &tmK, BAR(K_FULL), kvh * HD + bx * 64, j0, b);
            bool ok = true;
            if constexpr (kDK) {
                // V through the Q ring's space (both stages) into TMEM, before the first tiles
                if (elect_one()) mbar_expect_tx(BAR(V_FULL), kKBytes);
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx)
                    if (elect_one())
                        tma_load_3d(sbase + kRingOff + bx * (BKV * 128), &tmV, BAR(V_FULL), kvh * HD + bx * 64, j0, b);
                ok = warp_wait(BAR(V_COPIED), 0, P.status, ST_BWD_PRODUCER, &abort_flag);
            }
            int nq = 0, ngo = 0;  // Q and dO tiles issued
            for (int n = 0; ok && n < ntiles; ++n) {
                const int s = n % NS, use = n / NS;
                const int h = tile_head(n), i0 = tile_i0(n);
                // -LSE*log2(e) and -D of these 64 rows (padded rows: -inf and 0), with the
                // ring released last
                auto stats = [&](int bar) {
                    const long long srow = ((long long)b * P.H + h) * P.tq_pad + i0;
                    const uint32_t sdst = sbase + kStatOff + s * kStatBytes;
                    if (elect_one()) bulk_load(sdst, P.nlse2 + srow, BQ * 4, BAR(bar));
                    if (elect_one()) bulk_load(sdst + BQ * 4, P.ndelta + srow, BQ * 4, BAR(bar));
                };
                if (use > 0 && !warp_wait(BAR(Q_EMPTY(s)), (use - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) mbar_expect_tx(BAR(Q_FULL(s)), kTBytes + (kDK ? kStatBytes : 0));
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx)
                    if (elect_one())
                        tma_load_3d(sbase + kRingOff + s * kTBytes + bx * (BQ * 128), &tmQ, BAR(Q_FULL(s)),
                                    h * HD + bx * 64, i0, b);
                if (kDK) stats(Q_FULL(s));
                nq = n + 1;
                if (use > 0 && !warp_wait(BAR(G_EMPTY(s)), (use - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) mbar_expect_tx(BAR(G_FULL(s)), kTBytes + (kDK ? 0 : kStatBytes));
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx)
                    if (elect_one())
                        tma_load_3d(sbase + kGRingOff + s * kTBytes + bx * (BQ * 128), &tmG, BAR(G_FULL(s)),
                                    h * HD + bx * 64, i0, b);
                if (!kDK) stats(G_FULL(s));
                ngo = n + 1;
            }
            // every copy in flight lands before the CTA exits
            mbar_wait(BAR(K_FULL), 0, P.status, ST_TEARDOWN, nullptr);
            if (kDK) mbar_wait(BAR(V_FULL), 0, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, nq - NS); n < nq; ++n)
                mbar_wait(BAR(Q_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, ngo - NS); n < ngo; ++n)
                mbar_wait(BAR(G_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
        }
    } else if (warp == 5) {
        // ---------------------------------------------- MMA issuer (whole warp)
        if (ntiles > 0) {
            constexpr uint32_t idS = idesc_f16(BF16, BKV, BQ, false, false);
            constexpr uint32_t idAcc = idesc_f16(BF16, BKV, HD, false, true);
            auto wait_all = [&](int bar, uint32_t parity) -> bool {
                return warp_wait(BAR(bar), parity, P.status, ST_BWD_MMA, &abort_flag);
            };
            bool ok = wait_all(K_FULL, 0);
            if (kDK && ok) ok = wait_all(V_COPIED, 0);
            // S^T (and, in the dK pass, dP^T) of tile n: buffer n & 1 in the dV pass, the
            // single one in the dK pass
            auto issue_s = [&](int n) -> bool {
                const int s = n % NS, bf = kDK ? 0 : (n & 1);
                if (!wait_all(Q_FULL(s), (n / NS) & 1)) return false;
                if (kDK && !wait_all(G_FULL(s), (n / NS) & 1)) return false;
                tc_fence_after();
                const uint32_t qa = sbase + kRingOff + s * kTBytes, ga = sbase + kGRingOff + s * kTBytes;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * (BKV * 128) + (kk & 3) * 32;
                    const uint32_t boff = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
                    mma_ss_e(tbase + bf * 64, sdesc_sw128(sbase + kKOff + aoff, 16, 1024),
                               sdesc_sw128(qa + boff, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
                if constexpr (kDK) {
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t boff = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
                        mma_ts_e(tbase + 64, tV + kk * 8, sdesc_sw128(ga + boff, 16, 1024), idS, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit_e(BAR(ST_FULL(bf)));
                // the tile's ring read only by these MMAs is free once they complete
                mma_commit_e(BAR(kDK ? G_EMPTY(s) : Q_EMPTY(s)));
                return true;
            };
            if (ok) ok = issue_s(0);
            if (!kDK && ok && ntiles > 1) ok = issue_s(1);
            for (int n = 0; ok && n < ntiles; ++n) {
                const int s = n % NS, bf = kDK ? 0 : (n & 1);
                if (!wait_all(PT_FULL(bf), kDK ? (n & 1) : ((n >> 1) & 1)) ||
                    (!kDK && !wait_all(G_FULL(s), (n / NS) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dV += P^T dO, or dK += dS^T Q: the 16-bit operand over the first 32
                // columns of the S^T buffer, B = the tile's dO (Q) as [query][hd]
                const uint32_t bsrc = kDK ? sbase + kRingOff + s * kTBytes : sbase + kGRingOff + s * kTBytes;
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts_e(tAcc, tbase + bf * 64 + kk * 8, sdesc_sw128(bsrc + kk * 2048, BQ * 128, 1024), idAcc,
                               (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit_e(BAR(kDK ? Q_EMPTY(s) : G_EMPTY(s)));
                const int nx = kDK ? n + 1 : n + 2;
                if (nx < ntiles) ok = issue_s(nx);
            }
            if (ok) mma_commit_e(BAR(ACC_DONE));
            mma_commit_e(BAR(MMA_DONE));
            mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
        }
    } else {
        // ------------------------------------------- compute: one key row per thread
        const int r = warp * 32 + lane;
        const int j = j0 + r;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const bool key_live = j < P.Tk && (!P.key_mask || P.key_mask[(long long)b * P.mask_bstride + j] > 0.5f);
        auto wait_warp = [&](int bar, uint32_t parity) -> bool {
            const bool rr = mbar_wait(BAR(bar), parity, P.status, ST_BWD_COMPUTE, &abort_flag);
            return __all_sync(0xffffffffu, rr);
        };
        bool ok = true;
        if (kDK && ntiles > 0) {
            // V of the key block into TMEM: this thread's row, four 64-column boxes
            ok = wait_warp(V_FULL, 0);
            if (ok) {
#pragma unroll 1
                for (int bx = 0; bx < kBoxes; ++bx) {
                    uint32_t wv[32];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(smem + kRingOff + bx * (BKV * 128) + r * 128 +
                                                                         ((ch ^ (r & 7)) << 4));
                        wv[4 * ch] = v4.x;
                        wv[4 * ch + 1] = v4.y;
                        wv[4 * ch + 2] = v4.z;
                        wv[4 * ch + 3] = v4.w;
                    }
                    tmem_st32(tV + lane_off + bx * 32, wv);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(V_COPIED));  // the Q ring's space may be reloaded
            }
        }
        for (int n = 0; ok && n < ntiles; ++n) {
            const int s = n % NS, bf = kDK ? 0 : (n & 1);
            const int i0 = tile_i0(n);
            // visible query columns of this key row: [clo, chi); query position p sees
            // key j when p - wl <= j <= p + wr
            int clo = 0, chi = min(BQ, P.Tq - i0);
            if (P.wr >= 0) clo = max(clo, j - P.wr - P.q_offset - i0);
            if (P.wl >= 0) chi = min(chi, j + P.wl - P.q_offset - i0 + 1);
            if (!key_live) chi = 0;
            // the stats arrive with the tile's later-released ring; S^T (dP^T) come from the MMA
            if (!wait_warp(L_FULL(s), (n / NS) & 1) ||
                !wait_warp(ST_FULL(bf), kDK ? (n & 1) : ((n >> 1) & 1))) {
                ok = false;
                break;
            }
            const float* st_l = stat + s * 2 * BQ;
            const float* st_d = st_l + BQ;
            tc_fence_after();
            uint32_t sv[2][32], dp[kDK ? 2 : 1][32];
            tmem_ld32(tbase + lane_off + bf * 64, sv[0]);
            tmem_ld32(tbase + lane_off + bf * 64 + 32, sv[1]);
            if constexpr (kDK) {
                tmem_ld32(tbase + lane_off + 64, dp[0]);
                tmem_ld32(tbase + lane_off + 96, dp[1]);
            }
            tmem_ld_wait_only();
            tmem_pin(sv[0]);
            tmem_pin(sv[1]);
            if constexpr (kDK) {
                tmem_pin(dp[0]);
                tmem_pin(dp[1]);
            }
            // invisible pairs become -inf (P = 0)
            if (!__all_sync(0xffffffffu, clo <= 0 && chi >= BQ)) {
#pragma unroll
                for (int cc = 0; cc < BQ; ++cc)
                    sv[cc >> 5][cc & 31] = (cc >= clo && cc < chi) ? sv[cc >> 5][cc & 31] : 0xff800000u;
            }
            // P^T (dV pass) or dS^T = P^T (dP^T - D) (1 - tanh^2) (dK pass), as 16-bit
            // pairs over the first 32 columns of the S^T buffer
            uint32_t pk[32];
#pragma unroll
            for (int cc = 0; cc < BQ; cc += 2) {
                float d0, d1;
                const float p0 = b256_p<kCap>(P, __uint_as_float(sv[cc >> 5][cc & 31]), st_l[cc], d0);
                const float p1 = b256_p<kCap>(P, __uint_as_float(sv[cc >> 5][(cc & 31) + 1]), st_l[cc + 1], d1);
                if constexpr (kDK) {
                    const float g0 = p0 * (__uint_as_float(dp[cc >> 5][cc & 31]) + st_d[cc]) * d0;
                    const float g1 = p1 * (__uint_as_float(dp[cc >> 5][(cc & 31) + 1]) + st_d[cc + 1]) * d1;
                    pk[cc >> 1] = pack2<BF16>(g0, g1);
                } else {
                    pk[cc >> 1] = pack2<BF16>(p0, p1);
                }
            }
            tmem_st32(tbase + lane_off + bf * 64, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(PT_FULL(bf)));
        }
        // epilogue: dV, or dK * scale, of this key row (zero when no query sees the block)
        const bool have = ok && ntiles > 0 && wait_warp(ACC_DONE, 0);
        if (have) tc_fence_after();
        if (have || (ok && ntiles == 0)) {
            const float mul = kDK ? P.scale : 1.f;
            uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(kDK ? P.dk : P.dv) +
                                                  (((long long)b * P.Tk + j) * P.Hkv + kvh) * HD);
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t acc[32];
                if (have) {
                    tmem_ld32(tAcc + lane_off + c * 32, acc);
                    tmem_ld_wait(acc);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = 0u;
                }
                uint32_t q[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    q[e] = pack2<BF16>(__uint_as_float(acc[2 * e]) * mul, __uint_as_float(acc[2 * e + 1]) * mul);
                if (j < P.Tk) {
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) row[c * 4 + w4] = make_uint4(q[4 * w4], q[4 * w4 + 1], q[4 * w4 + 2], q[4 * w4 + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// dQ of 128 query rows of one (b, h).  MODE 0: dense; MODE 4: with a softcap.
template <bool BF16, int MODE>
__global__ void __launch_bounds__(b256::kThreads, 1)
    bwd_h256_dq_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG) {
    using namespace b256;
    constexpr bool kCap = (MODE & 4) != 0;
    constexpr int NS = kDqStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDqBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kDqNumBars);
    __shared__ int abort_flag;
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int Q_FULL = 0;     // Q in ring stage 0
    const int Q_COPIED = 1;   // ... copied into TMEM (4 compute warps)
    const int G_FULL = 2;     // dO in shared memory
    const int ACC_DONE = 3;
    const int MMA_DONE = 4;
    const int SD_FULL = 5;    // S and dP of a tile in TMEM
    const int DS_FULL = 6;    // dS of a tile in TMEM (4 compute warps)
    auto KV_FULL = [&](int s) { return 7 + s; };
    auto KV_EMPTY = [&](int s) { return 7 + NS + s; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // query blocks longest first (causally the last see the most keys), every head's
    // block qb before any one's block qb - 1
    const int nqb = (P.Tq + BQD - 1) / BQD, nh = P.H * P.B;
    const int qb = nqb - 1 - (int)blockIdx.x / nh, hb = (int)blockIdx.x % nh;
    const int h = hb % P.H, b = hb / P.H, kvh = h / P.G;
    const int i0 = qb * BQD;
    const int prow0 = i0 + P.q_offset, prow1 = min(i0 + BQD, P.Tq) - 1 + P.q_offset;
    int klo, khi;
    key_range(P.wl, P.wr, P.Tk, prow0, prow1, &klo, &khi);
    const int t0 = klo / BKD;
    const int nkt = khi > klo ? (khi + BKD - 1) / BKD - t0 : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDqNumBars; ++i) mbar_init(BAR(i), (i == Q_COPIED || i == DS_FULL) ? 4 : 1);
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
    const uint32_t tS = tbase, tDP = tbase + 64, tQ = tbase + 128, tDQ = tbase + 256;

    if (warp == 4) {
        // ---------------------------------------------- TMA producer (whole warp)
        if (nkt > 0) {
            if (elect_one()) {
                prefetch_tmap(&tmQ);
                prefetch_tmap(&tmK);
                prefetch_tmap(&tmV);
                prefetch_tmap(&tmG);
            }
            if (elect_one()) mbar_expect_tx(BAR(Q_FULL), BQD * HD * 2);
            if (elect_one()) mbar_expect_tx(BAR(G_FULL), kDoBytes);
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx) {
                if (elect_one())
                    tma_load_3d(sbase + kDqRingOff + bx * (BQD * 128), &tmQ, BAR(Q_FULL), h * HD + bx * 64, i0, b);
                if (elect_one())
                    tma_load_3d(sbase + kDoOff + bx * (BQD * 128), &tmG, BAR(G_FULL), h * HD + bx * 64, i0, b);
            }
            // K and V tiles go into the ring once Q has left stage 0 for TMEM
            bool ok = warp_wait(BAR(Q_COPIED), 0, P.status, ST_BWD_PRODUCER, &abort_flag);
            int issued = 0;
            for (int n = 0; ok && n < nkt; ++n) {
                const int s = n % NS, use = n / NS;
                if (use > 0 && !warp_wait(BAR(KV_EMPTY(s)), (use - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag))
                    break;
                const int j0 = (t0 + n) * BKD;
                const uint32_t ka = sbase + kDqRingOff + s * 2 * kKTileBytes, va = ka + kKTileBytes;
                if (elect_one()) mbar_expect_tx(BAR(KV_FULL(s)), 2 * kKTileBytes);
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx) {
                    if (elect_one()) tma_load_3d(ka + bx * (BKD * 128), &tmK, BAR(KV_FULL(s)), kvh * HD + bx * 64, j0, b);
                    if (elect_one()) tma_load_3d(va + bx * (BKD * 128), &tmV, BAR(KV_FULL(s)), kvh * HD + bx * 64, j0, b);
                }
                issued = n + 1;
            }
            // every copy in flight lands before the CTA exits
            mbar_wait(BAR(Q_FULL), 0, P.status, ST_TEARDOWN, nullptr);
            mbar_wait(BAR(G_FULL), 0, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, issued - NS); n < issued; ++n)
                mbar_wait(BAR(KV_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
        }
    } else if (warp == 5) {
        // ---------------------------------------------- MMA issuer (whole warp)
        if (nkt > 0) {
            constexpr uint32_t idS = idesc_f16(BF16, BQD, BKD, false, false);
            constexpr uint32_t idAcc = idesc_f16(BF16, BQD, HD, false, true);
            auto wait_all = [&](int bar, uint32_t parity) -> bool {
                return warp_wait(BAR(bar), parity, P.status, ST_BWD_MMA, &abort_flag);
            };
            bool ok = wait_all(Q_COPIED, 0) && wait_all(G_FULL, 0);
            // S = Q K^T (A from TMEM) and dP = dO V^T (both operands in shared memory)
            auto issue_sd = [&](int n) -> bool {
                const int s = n % NS;
                if (!wait_all(KV_FULL(s), (n / NS) & 1)) return false;
                tc_fence_after();
                const uint32_t ka = sbase + kDqRingOff + s * 2 * kKTileBytes, va = ka + kKTileBytes;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t boff = (kk >> 2) * (BKD * 128) + (kk & 3) * 32;
                    mma_ts_e(tS, tQ + kk * 8, sdesc_sw128(ka + boff, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * (BQD * 128) + (kk & 3) * 32;
                    const uint32_t boff = (kk >> 2) * (BKD * 128) + (kk & 3) * 32;
                    mma_ss_e(tDP, sdesc_sw128(sbase + kDoOff + aoff, 16, 1024), sdesc_sw128(va + boff, 16, 1024), idS,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit_e(BAR(SD_FULL));
                return true;
            };
            if (ok) ok = issue_sd(0);
            for (int n = 0; ok && n < nkt; ++n) {
                const int s = n % NS;
                if (!wait_all(DS_FULL, n & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dQ += dS K: dS as 16-bit pairs over the first 32 columns of S, B = K as [key][hd]
                const uint32_t ka = sbase + kDqRingOff + s * 2 * kKTileBytes;
#pragma unroll
                for (int kk = 0; kk < BKD / 16; ++kk)
                    mma_ts_e(tDQ, tS + kk * 8, sdesc_sw128(ka + kk * 2048, BKD * 128, 1024), idAcc,
                               (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit_e(BAR(KV_EMPTY(s)));
                if (n + 1 < nkt) ok = issue_sd(n + 1);
            }
            if (ok) mma_commit_e(BAR(ACC_DONE));
            mma_commit_e(BAR(MMA_DONE));
            mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
        }
    } else {
        // ------------------------------------------ compute: one query row per thread
        const int r = warp * 32 + lane;
        const int i = i0 + r;
        const int p = i + P.q_offset;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        auto wait_warp = [&](int bar, uint32_t parity) -> bool {
            const bool rr = mbar_wait(BAR(bar), parity, P.status, ST_BWD_COMPUTE, &abort_flag);
            return __all_sync(0xffffffffu, rr);
        };
        // -LSE*log2(e) and -D of this row (rows past the last query see no key)
        const long long srow = ((long long)b * P.H + h) * P.tq_pad + i;
        const float nl = i < P.Tq ? P.nlse2[srow] : -INFINITY;
        const float nd = i < P.Tq ? P.ndelta[srow] : 0.f;
        bool ok = true;
        if (nkt > 0) {
            // Q into TMEM: this thread's row, four 64-column boxes
            ok = wait_warp(Q_FULL, 0);
            if (ok) {
#pragma unroll 1
                for (int bx = 0; bx < kBoxes; ++bx) {
                    uint32_t wv[32];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(smem + kDqRingOff + bx * (BQD * 128) + r * 128 +
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
                if (lane == 0) mbar_arrive(BAR(Q_COPIED));
            }
        }
        for (int n = 0; ok && n < nkt; ++n) {
            const int j0 = (t0 + n) * BKD;
            uint32_t mbits[2] = {0xffffffffu, 0xffffffffu};
            if (P.key_mask) {
                const float* mrow = P.key_mask + (long long)b * P.mask_bstride;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int j = j0 + c * 32 + lane;
                    mbits[c] = __ballot_sync(0xffffffffu, j < P.Tk && mrow[j] > 0.5f);
                }
            }
            const bool full =
                tile_full(P.wl, P.wr, P.Tk, prow0, prow1, j0, j0 + BKD) && (mbits[0] & mbits[1]) == 0xffffffffu;
            int clo = 0, chi = BKD;
            if (!full) {
                chi = min(chi, P.Tk - j0);
                if (P.wr >= 0) chi = min(chi, p + P.wr - j0 + 1);
                if (P.wl >= 0) clo = max(clo, p - P.wl - j0);
                if (i >= P.Tq) chi = 0;
            }
            if (!wait_warp(SD_FULL, n & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[2][32], dp[2][32];
            tmem_ld32(tS + lane_off, sv[0]);
            tmem_ld32(tS + lane_off + 32, sv[1]);
            tmem_ld32(tDP + lane_off, dp[0]);
            tmem_ld32(tDP + lane_off + 32, dp[1]);
            tmem_ld_wait_only();
            tmem_pin(sv[0]);
            tmem_pin(sv[1]);
            tmem_pin(dp[0]);
            tmem_pin(dp[1]);
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
            // dS = P (dP - D) (1 - tanh^2) as 16-bit pairs over the first 32 columns of S
            uint32_t pk[32];
#pragma unroll
            for (int cc = 0; cc < BKD; cc += 2) {
                float d0, d1;
                const float p0 = b256_p<kCap>(P, __uint_as_float(sv[cc >> 5][cc & 31]), nl, d0);
                const float p1 = b256_p<kCap>(P, __uint_as_float(sv[cc >> 5][(cc & 31) + 1]), nl, d1);
                const float g0 = p0 * (__uint_as_float(dp[cc >> 5][cc & 31]) + nd) * d0;
                const float g1 = p1 * (__uint_as_float(dp[cc >> 5][(cc & 31) + 1]) + nd) * d1;
                pk[cc >> 1] = pack2<BF16>(g0, g1);
            }
            tmem_st32(tS + lane_off, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(DS_FULL));
        }
        // epilogue: dQ * scale of this row (zero when it sees no key)
        const bool have = ok && nkt > 0 && wait_warp(ACC_DONE, 0);
        if (have) tc_fence_after();
        if (have || (ok && nkt == 0)) {
            uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(P.dq) +
                                                  (((long long)b * P.Tq + i) * P.H + h) * HD);
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t acc[32];
                if (have) {
                    tmem_ld32(tDQ + lane_off + c * 32, acc);
                    tmem_ld_wait(acc);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = 0u;
                }
                uint32_t q[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    q[e] = pack2<BF16>(__uint_as_float(acc[2 * e]) * P.scale, __uint_as_float(acc[2 * e + 1]) * P.scale);
                if (i < P.Tq) {
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) row[c * 4 + w4] = make_uint4(q[4 * w4], q[4 * w4 + 1], q[4 * w4 + 2], q[4 * w4 + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// Passes as for the other head sizes (1: D and -LSE*log2(e) into the workspace, 2:
// dK/dV, 4: dQ).  Both tensor-core passes read D from the workspace, so pass 4 runs
// the preprocess too; dK and dV take one launch each.
template <bool BF16>
cudaError_t bwd_hd256_typed(const Params& p, const BwdMaps& m, int phases, cudaStream_t s) {
    cudaError_t e;
    const bool c = p.softcap > 0.f;
    if (phases & 5) {
        e = launch_bwd_preprocess(p, BF16 ? 2 : 1, s);
        if (e != cudaSuccess) return e;
    }
    if (phases & 2) {
        auto kdv = c ? bwd_h256_kv_kernel<BF16, 4, 1> : bwd_h256_kv_kernel<BF16, 0, 1>;
        auto kdk = c ? bwd_h256_kv_kernel<BF16, 4, 2> : bwd_h256_kv_kernel<BF16, 0, 2>;
        if ((e = cudaFuncSetAttribute(kdv, cudaFuncAttributeMaxDynamicSharedMemorySize, b256::kKVLaunchBytes)) !=
                cudaSuccess ||
            (e = cudaFuncSetAttribute(kdk, cudaFuncAttributeMaxDynamicSharedMemorySize, b256::kKVLaunchBytes)) !=
                cudaSuccess)
            return e;
        const unsigned grid = (unsigned)((p.Tk + b256::BKV - 1) / b256::BKV) * p.Hkv * p.B;
        kdv<<<grid, b256::kThreads, b256::kKVLaunchBytes, s>>>(p, m.q64, m.k, m.v, m.dout64);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        kdk<<<grid, b256::kThreads, b256::kKVLaunchBytes, s>>>(p, m.q64, m.k, m.v, m.dout64);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (phases & 4) {
        auto kdq = c ? bwd_h256_dq_kernel<BF16, 4> : bwd_h256_dq_kernel<BF16, 0>;
        if ((e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, b256::kDqLaunchBytes)) !=
            cudaSuccess)
            return e;
        const unsigned grid = (unsigned)((p.Tq + b256::BQD - 1) / b256::BQD) * p.H * p.B;
        kdq<<<grid, b256::kThreads, b256::kDqLaunchBytes, s>>>(p, m.q, m.k64, m.v64, m.dout);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

}  // namespace attn
