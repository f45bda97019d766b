// bwd_tc.cuh -- FlashAttention-2-style backward on the tcgen05 tensor cores.
//
// Deterministic and free of atomics: one kernel owns dK/dV of a 128-key block
// (summing over the GQA group's query heads in TMEM), a second owns dQ of a
// 128-row query block.  Both recompute P = exp(st - LSE) from the saved LSE.
// Sources: vision_rs flash_attn2.rs, "Backward - dQ" and "Backward - dK / dV"
// (p = exp(s*scale - L), dS = p (dO.V - D), dQ += dS K scale, dK += dS Q scale,
// dV += p dO); forge attention.metal, attention_bwd_dq_f32 / attention_bwd_dkv_f32
// (softcap derivative 1 - tanh^2 of the uncapped score, dK/dV summed over
// the query heads sharing a KV head, no atomics); ferrotensor
// engine/attention.rs, flash_attention_v2_backward_with (a dQ pass over query
// tiles and a dK/dV pass over key tiles, 128 rows each).
//
// dK/dV kernel: CTA = 128 keys of one (b, kv head), 6 warps.
//   warp 4  TMA: K and V once, then 64-row Q and dO tiles of every query head
//           of the group into a ring.
//   warp 5  MMA (one thread): S^T = K Q^T and dP^T = V dO^T into a double
//           buffer; after the compute warps turn them into P^T and dS^T
//           (16-bit, written over the first half of each buffer):
//           dV += P^T dO and dK += dS^T Q, A operand from TMEM.
//   warps 0-3  one thread per key row: P^T = exp2(st*log2e - LSE*log2e) on
//           visible pairs, dS^T = P^T (dP^T - D) (* (1 - tanh^2)).
//   TMEM: S^T 0/64, dP^T 128/192, dV 256, dK 256+hd.
// dQ kernel: CTA = 128 query rows of one (b, h): S = Q K^T and dP = dO V^T
//   over 64-key tiles (double buffer), dS written over S, dQ += dS K.  Q and
//   dO are copied once into TMEM so all three GEMMs take A from TMEM.
//   TMEM: S 0/64, dP 128/192, dQ 256, Q 256+hd, dO 256+hd+hd/2.
#include <math.h>

#include <algorithm>
#include <type_traits>

#pragma once

#include "kernels.h"

namespace attn {
namespace {

// dK/dV: compute warps (four, one key row per thread; eight with a softcap, two
// per key row splitting each tile's query columns), then the producer and the MMA warp
__host__ __device__ constexpr int dkdv_compute_warps(int mode) { return (mode & 4) ? 8 : 4; }
__host__ __device__ constexpr int dkdv_threads(int mode) { return 32 * (dkdv_compute_warps(mode) + 2); }
constexpr int kThreadsDQ = 384;
// dQ registers: the eight compute warps take 184, the producers and MMA issuers 136
// (256*184 + 128*136 = 64512 = 384 threads at launch * 168)
constexpr int kDqRegsCompute = 184, kDqRegsAux = 136;
static_assert(256 * kDqRegsCompute + 128 * kDqRegsAux <= kThreadsDQ * 168, "register split exceeds launch");  // dQ: 8 compute warps, K/V producer, two MMA issuers, Q/dO/O producer
constexpr float kLog2e = 1.4426950408889634f;

// TMEM column (within a 64-column tile buffer) of K-step kk's 16-bit dS operand
// in the dQ kernel: the two compute warps of a row each pack their 32 columns
// into the first 16 of them, so the 32 operand columns sit at 0..15 and 32..47.
__device__ __forceinline__ uint32_t pcol(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

// =============================================================== dK / dV
template <int HD>
struct KVCfg {
    static constexpr int BKV = 128;  // keys per CTA
    static constexpr int BQ = 64;    // query rows per inner tile
    static constexpr int kBoxes = HD / 64;
    static constexpr int kStages = 4;
    static constexpr int kKVBytes = BKV * HD * 2;
    static constexpr int kQBytes = BQ * HD * 2;  // one Q (or dO) tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKVBytes;
    static constexpr int kQOff = 2 * kKVBytes;
    static constexpr int kGOff = kQOff + kStages * kQBytes;   // dO ring
    static constexpr int kStatOff = kGOff + kStages * kQBytes;  // [stage][2][BQ] floats: -LSE*log2e, -D
    static constexpr int kStatBytes = 2 * BQ * 4;
    static constexpr int kBarOff = kStatOff + kStages * kStatBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1 + 1 + 1;
    // epilogue staging: 32-row x 64-column slices of 4 KB, two per compute warp
    // (one with eight compute warps)
    static constexpr int kStgOff = kQOff;  // the Q ring, free once every tile's MMAs completed
    static constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
    static constexpr int kLaunchBytes = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
    static_assert(kStages * kQBytes >= 8 * 4096, "staging fits in the Q ring");
};

// MODE & 3 -- 0: dense; 1: packed variable-length sequences (cu_seqlens); 2: dense with
// an additive score bias; MODE & 4: softcap; MODE & 8: a head size below HD through
// 4-D maps (the columns past the head load as zeros and are never stored); MODE 64:
// packed fused-QKV rows of one batch, each row limited to its own sequence.  Each
// instantiation carries only its own bookkeeping (the softcap's registers, live through
// the tile loop, made the plain path spill when it was a run-time branch).
template <bool BF16, int HD, int MODE>
__global__ void __launch_bounds__(dkdv_threads(MODE), 1)
    bwd_dkdv_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV) {
    using C = KVCfg<HD>;
    constexpr int NS = C::kStages, BQ = C::BQ, BKV = C::BKV;
    constexpr int NCW = dkdv_compute_warps(MODE), HF = NCW / 4;  // HF warps per key row
    constexpr int PRODUCER = NCW, MMA = NCW + 1;
    constexpr bool VL = (MODE & 3) == 1, BIAS = (MODE & 3) == 2, PADH = (MODE & 8) != 0;
    constexpr bool RB = (MODE & 64) != 0;  // packed fused-QKV rows: per-row sequence bounds
    static_assert(!RB || MODE == 64, "the row bounds are built for dense batches without other modes");
    static_assert(!(PADH && VL), "padded head sizes are built for dense batches only");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    float* stat = reinterpret_cast<float*>(smem + C::kStatOff);
    __shared__ int abort_flag;
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int KV_FULL = 0;
    auto Q_FULL = [&](int s) { return 1 + s; };
    auto Q_EMPTY = [&](int s) { return 1 + NS + s; };
    auto ST_FULL = [&](int b) { return 1 + 2 * NS + b; };
    auto PT_FULL = [&](int b) { return 3 + 2 * NS + b; };
    const int ACC_DONE = 5 + 2 * NS;
    const int MMA_DONE = 6 + 2 * NS;
    const int LD_DONE = 7 + 2 * NS;  // the compute warps have read S^T/dP^T of a tile (HF = 2)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1-D grid over chunks of kv_chunk (batch, KV head) pairs, and inside a chunk key
    // blocks longest first (causally the first key blocks are seen by the most
    // queries): the CTAs that stream the same Q and dO tiles run together while L2
    // still holds them, and the light blocks of one chunk overlap the next chunk
    const int ng = P.Hkv * P.B, nkb = (int)gridDim.x / ng;
    const int CH = P.kv_chunk > 0 ? min(P.kv_chunk, ng) : ng;
    const int cidx = (int)blockIdx.x / (nkb * CH), ch = min(CH, ng - cidx * CH);
    const int within = (int)blockIdx.x - cidx * nkb * CH;
    const int kg = cidx * CH + within % ch;
    const int kvh = kg % P.Hkv, b = kg / P.Hkv;
    // (packed fused-QKV rows: key blocks heaviest first, when an order is given)
    const int j0 = (RB && P.item_order ? __ldg(P.item_order + within / ch) : within / ch) * BKV;
    const Seq sq = seq_of<VL>(P, b);
    if (j0 >= sq.tk) return;  // (packed) past this sequence's keys: nothing to write
    int qlo, qhi;
    query_range(P.wl, P.wr, sq.tq, P.q_offset, j0, min(j0 + BKV, sq.tk), &qlo, &qhi);
    if constexpr (RB) {  // packed fused-QKV rows: a key is seen only from its own sequence
        qlo = max(qlo, row_keys(P, j0, sq.tq).x);
        qhi = max(qlo, min(qhi, row_keys(P, min(j0 + BKV, sq.tk) - 1, sq.tq).y));
    }
    const int qt0 = qlo / BQ;
    const int nqt = qhi > qlo ? (qhi + BQ - 1) / BQ - qt0 : 0;
    const int ntiles = nqt * P.G;  // (head, query tile) pairs, head-major
    auto tile_head = [&](int n) { return kvh * P.G + n / max(nqt, 1); };
    auto tile_i0 = [&](int n) { return (qt0 + n % max(nqt, 1)) * BQ; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i)
            mbar_init(BAR(i), (i == PT_FULL(0) || i == PT_FULL(1) || i == LD_DONE) ? NCW : 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == MMA) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tDV = tbase + 256, tDK = tbase + 256 + HD;

    if (warp == PRODUCER) {
        // producer and MMA issuer run as whole warps; one elected lane issues
        if (ntiles > 0) {
            if (elect_one()) {
                prefetch_tmap(&tmQ);
                prefetch_tmap(&tmK);
                prefetch_tmap(&tmV);
                prefetch_tmap(&tmG);
            }
            if (elect_one()) mbar_expect_tx(BAR(KV_FULL), 2 * C::kKVBytes);
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx) {
                if (elect_one())
                    tile_load<PADH, HD>(sbase + C::kKOff + bx * (BKV * 128), &tmK, BAR(KV_FULL), kvh, bx,
                                        sq.k0 + j0, sq.zb);
                if (elect_one())
                    tile_load<PADH, HD>(sbase + C::kVOff + bx * (BKV * 128), &tmV, BAR(KV_FULL), kvh, bx,
                                        sq.k0 + j0, sq.zb);
            }
            int issued = 0;
            for (int n = 0; n < ntiles; ++n) {
                const int s = n % NS, use = n / NS;
                if (use > 0 && !warp_wait(BAR(Q_EMPTY(s)), (use - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag))
                    break;
                const int h = tile_head(n), i0 = tile_i0(n);
                if (elect_one()) mbar_expect_tx(BAR(Q_FULL(s)), 2 * C::kQBytes + C::kStatBytes);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx) {
                    if (elect_one())
                        tile_load<PADH, HD>(sbase + C::kQOff + s * C::kQBytes + bx * (BQ * 128), &tmQ,
                                            BAR(Q_FULL(s)), h, bx, sq.q0 + i0, sq.zb);
                    if (elect_one())
                        tile_load<PADH, HD>(sbase + C::kGOff + s * C::kQBytes + bx * (BQ * 128), &tmG,
                                            BAR(Q_FULL(s)), h, bx, sq.q0 + i0, sq.zb);
                }
                // -LSE*log2(e) and -D of these 64 rows (padded rows: -inf and 0)
                const long long srow = ((long long)b * P.H + h) * P.tq_pad + i0;
                const uint32_t sdst = sbase + C::kStatOff + s * C::kStatBytes;
                if (elect_one()) bulk_load(sdst, P.nlse2 + srow, BQ * 4, BAR(Q_FULL(s)));
                if (elect_one()) bulk_load(sdst + BQ * 4, P.ndelta + srow, BQ * 4, BAR(Q_FULL(s)));
                issued = n + 1;
            }
            mbar_wait(BAR(KV_FULL), 0, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, issued - NS); n < issued; ++n)
                mbar_wait(BAR(Q_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
        }
    } else if (warp == MMA) {
        if (ntiles > 0) {
            constexpr uint32_t idS = idesc_f16(BF16, BKV, BQ, false, false);
            constexpr uint32_t idAcc = idesc_f16(BF16, BKV, HD, false, true);
            bool ok = warp_wait(BAR(KV_FULL), 0, P.status, ST_BWD_MMA, &abort_flag);
            // S^T and dP^T of tile n into buffer n & 1
            auto issue_sd = [&](int n) -> bool {
                const int s = n % NS, bf = n & 1;
                if (!warp_wait(BAR(Q_FULL(s)), (n / NS) & 1, P.status, ST_BWD_MMA, &abort_flag)) return false;
                tc_fence_after();
                const uint32_t qa = sbase + C::kQOff + s * C::kQBytes, ga = sbase + C::kGOff + s * C::kQBytes;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * (BKV * 128) + (kk & 3) * 32;
                    const uint32_t boff = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
                    mma_ss_e(tbase + bf * 64, sdesc_sw128(sbase + C::kKOff + aoff, 16, 1024),
                               sdesc_sw128(qa + boff, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * (BKV * 128) + (kk & 3) * 32;
                    const uint32_t boff = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
                    mma_ss_e(tbase + 128 + bf * 64, sdesc_sw128(sbase + C::kVOff + aoff, 16, 1024),
                               sdesc_sw128(ga + boff, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
                mma_commit_e(BAR(ST_FULL(bf)));
                return true;
            };
            if (ok) ok = issue_sd(0);
            if (ok && ntiles > 1) ok = issue_sd(1);
            for (int n = 0; ok && n < ntiles; ++n) {
                const int s = n % NS, bf = n & 1;
                if (!warp_wait(BAR(PT_FULL(bf)), (n >> 1) & 1, P.status, ST_BWD_MMA, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qa = sbase + C::kQOff + s * C::kQBytes, ga = sbase + C::kGOff + s * C::kQBytes;
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk) {
                    mma_ts_e(tDV, tbase + bf * 64 + kk * 8, sdesc_sw128(ga + kk * 2048, BQ * 128, 1024), idAcc,
                               (n > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk) {
                    mma_ts_e(tDK, tbase + 128 + bf * 64 + kk * 8, sdesc_sw128(qa + kk * 2048, BQ * 128, 1024),
                               idAcc, (n > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_e(BAR(Q_EMPTY(s)));
                if (n + 2 < ntiles) ok = issue_sd(n + 2);
            }
            if (ok) mma_commit_e(BAR(ACC_DONE));
            mma_commit_e(BAR(MMA_DONE));
            mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
        }
    } else {
        // ------------ compute: warp w owns TMEM lane quarter w % 4 (one key row per
        // thread); with HF = 2, warps w and w+4 split each tile's 64 query columns (hf)
        const int wq = warp & 3, hf = warp >> 2;
        const int r = wq * 32 + lane;
        const int j = j0 + r;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const bool key_live = j < sq.tk && (!P.key_mask || P.key_mask[(long long)b * P.mask_bstride + j] > 0.5f);
        int2 rk_key = make_int2(0, sq.tq);  // packed fused-QKV rows: this key's sequence
        if constexpr (RB) rk_key = row_keys(P, max(min(j, sq.tk - 1), 0), sq.tq);
        constexpr bool cap = (MODE & 4) != 0;
        constexpr int kc = BQ / HF;  // query columns per thread
        const float cap_in = P.scale / fmaxf(P.softcap, 1e-30f);
        const uint64_t sl2_2 = f2_make(P.scale_log2, P.scale_log2), one2 = f2_make(1.f, 1.f);
        bool ok = true;
        for (int n = 0; n < ntiles; ++n) {
            const int bf = n & 1;
            const int h = tile_head(n), i0 = tile_i0(n);
            const int c0 = kc * hf;  // this thread's first query column of the tile
            // visible query columns of this key row among the thread's: [clo, chi)
            int clo = 0, chi = min(kc, sq.tq - i0 - c0);
            // query position p sees key j when p - wl <= j <= p + wr
            if (P.wr >= 0) clo = max(clo, j - P.wr - P.q_offset - i0 - c0);
            if (P.wl >= 0) chi = min(chi, j + P.wl - P.q_offset - i0 - c0 + 1);
            if constexpr (RB) {  // packed fused-QKV rows: the queries of this key's sequence
                clo = max(clo, rk_key.x - i0 - c0);
                chi = min(chi, rk_key.y - i0 - c0);
            }
            if (!key_live) chi = 0;
            // additive score bias of (query i0 + c0 + cc, key j): the
            // first 32 columns' loads issue before the waits; rows past the last query read
            // the last row (finite; those columns are masked below), so the loads issue
            // back to back without a branch
            const float* bcol = BIAS ? P.bias + (long long)b * P.bias_sb + (long long)h * P.bias_sh +
                                           (long long)(key_live ? j : 0) * P.bias_sk
                                     : nullptr;
            const int ilast = max(sq.tq - 1, 0);
            float bv0[BIAS ? 32 : 1];
            if constexpr (BIAS) {
#pragma unroll
                for (int e = 0; e < 32; ++e) bv0[e] = __ldg(bcol + (long long)min(i0 + c0 + e, ilast) * P.bias_sq);
            }
            // the stats arrive with Q/dO of this tile; S^T/dP^T come from the MMA
            const int s = n % NS;
            if (!warp_wait(BAR(Q_FULL(s)), (n / NS) & 1, P.status, ST_BWD_COMPUTE, &abort_flag) ||
                !warp_wait(BAR(ST_FULL(bf)), (n >> 1) & 1, P.status, ST_BWD_COMPUTE, &abort_flag)) {
                ok = false;
                break;
            }
            const float* st_l = stat + s * 2 * BQ + c0;
            const float* st_d = st_l + BQ;
            tc_fence_after();
            uint32_t sv[kc], dp[kc];
            auto chunk = [](uint32_t* a, int c) -> uint32_t(&)[32] { return *reinterpret_cast<uint32_t(*)[32]>(a + 32 * c); };
#pragma unroll
            for (int c = 0; c < kc / 32; ++c) {
                tmem_ld32(tbase + lane_off + bf * 64 + c0 + 32 * c, chunk(sv, c));
                tmem_ld32(tbase + lane_off + 128 + bf * 64 + c0 + 32 * c, chunk(dp, c));
            }
            tmem_ld_wait_only();
#pragma unroll
            for (int c = 0; c < kc / 32; ++c) {
                tmem_pin(chunk(sv, c));
                tmem_pin(chunk(dp, c));
            }
            if constexpr (HF == 2) {
                // P^T and dS^T go over the first 32 columns of the buffers, which hold the
                // other warp's scores: both warps of a row must have read theirs first
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(LD_DONE));
            }
            // the bias joins the raw score here, or, with a softcap (which comes first), the
            // capped score inside the element loop (then kc = 32: bv0 holds the thread's columns)
            if constexpr (BIAS && !cap) {
                const float inv = 1.f / P.scale;
#pragma unroll
                for (int half = 0; half < kc / 32; ++half) {
                    float bv[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        bv[e] = half == 0 ? bv0[e]
                                          : __ldg(bcol + (long long)min(i0 + c0 + 32 * half + e, ilast) * P.bias_sq);
                    if (key_live)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            sv[32 * half + e] = __float_as_uint(fmaf(bv[e], inv, __uint_as_float(sv[32 * half + e])));
                }
            }
            uint32_t pk[kc / 2], dk[kc / 2];
            // With a softcap, the polynomial serves the warp's tile half unless a raw
            // score of its rows lies outside its range (checked before masking)
            bool poly = false, shorter = false;
            if (cap) {
                float amax = 0.f;
#pragma unroll
                for (int cc = 0; cc < kc; cc += 2)
                    amax = max3f(amax, fabsf(__uint_as_float(sv[cc])), fabsf(__uint_as_float(sv[cc + 1])));
                poly = __all_sync(0xffffffffu, amax <= cap_poly(P.scale, P.softcap).r_max);
                shorter = __all_sync(0xffffffffu, amax <= cap_short(P.scale, P.softcap).r_max);
            }
            // Where some pair is invisible, those scores become -inf first, so every tile
            // runs one copy of the element loop (a rarely run second copy would be fetched
            // into the instruction cache cold each time).
            const bool full = key_live && clo <= 0 && chi >= kc;
            if (!__all_sync(0xffffffffu, full)) {
#pragma unroll
                for (int cc = 0; cc < kc; ++cc) sv[cc] = (cc >= clo && cc < chi) ? sv[cc] : 0xff800000u;
                poly = poly && cap_poly(P.scale, P.softcap).inf_ok;
                shorter = shorter && cap_short(P.scale, P.softcap).inf_ok;
            }
            // Mode 0: no softcap; 1: softcap by the polynomial; 2: by tanh_accurate; 3: by
            // the short polynomial.  Pairs of columns go through the f32x2 unit together; the stats hold -LSE*log2e
            // and -D, so x = st*log2e + nl and dS = P*(dP + nd)*(1 - tanh^2).
            auto elems = [&](auto modec) {
                constexpr int kMode = decltype(modec)::value;
#pragma unroll
                for (int c = 0; c < kc; c += 2) {
                    const uint64_t nl = *reinterpret_cast<const uint64_t*>(st_l + c);
                    const uint64_t nd = *reinterpret_cast<const uint64_t*>(st_d + c);
                    const float s0 = __uint_as_float(sv[c]), s1 = __uint_as_float(sv[c + 1]);
                    const uint64_t dp2 = f2_make(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1]));
                    float p0, p1, x0, x1;
                    uint64_t dcap = one2;
                    // with a softcap, the bias (log2 units) joins after the cap
                    uint64_t nlb = nl;
                    if constexpr (BIAS && cap) nlb = f2_add(nl, f2_make(bv0[c] * kLog2e, bv0[c + 1] * kLog2e));
                    if constexpr (kMode == 2) {
                        // softcap*tanh(-inf) would be finite: keep a masked score at -inf
                        float l0, l1;
                        f2_split(nlb, l0, l1);
                        const float t0 = tanh_accurate(s0 * cap_in), t1 = tanh_accurate(s1 * cap_in);
                        x0 = s0 == -INFINITY ? -INFINITY : fmaf(P.softcap * kLog2e, t0, l0);
                        x1 = s1 == -INFINITY ? -INFINITY : fmaf(P.softcap * kLog2e, t1, l1);
                        dcap = f2_make(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
                    } else {
                        uint64_t g = f2_make(s0, s1);
                        if constexpr (kMode == 1) {
                            uint64_t uu;
                            const CapPoly cp = cap_poly(P.scale, P.softcap);
                            g = cap_g(cp, g, uu);
                            // 1 - tanh^2; a masked score gives g = -inf and -inf here, with P = 0
                            float d0, d1;
                            f2_split(f2_fma(f2_mul(g, g), cp.nc2, one2), d0, d1);
                            dcap = f2_make(fmaxf(d0, 0.f), fmaxf(d1, 0.f));
                        } else if constexpr (kMode == 3) {
                            // the short polynomial (every raw score of the tile within its range);
                            // a masked score gives g = -inf as above
                            g = cap_g_short(cap_short(P.scale, P.softcap), g);
                            float d0, d1;
                            f2_split(f2_fma(f2_mul(g, g), cap_poly(P.scale, P.softcap).nc2, one2), d0, d1);
                            dcap = f2_make(fmaxf(d0, 0.f), fmaxf(d1, 0.f));
                        }
                        f2_split(f2_fma(g, sl2_2, nlb), x0, x1);
                    }
                    p0 = fast_exp2(x0);
                    p1 = fast_exp2(x1);
                    const uint64_t pp = f2_make(p0, p1);
                    uint64_t ds = f2_mul(pp, f2_add(dp2, nd));
                    if constexpr (kMode != 0) ds = f2_mul(ds, dcap);
                    float q0, q1;
                    f2_split(ds, q0, q1);
                    pk[c >> 1] = pack2<BF16>(p0, p1);
                    dk[c >> 1] = pack2<BF16>(q0, q1);
                }
            };
            if (!cap) elems(std::integral_constant<int, 0>());
            else if (shorter) elems(std::integral_constant<int, 3>());
            else if (poly) elems(std::integral_constant<int, 1>());
            else elems(std::integral_constant<int, 2>());
            // 16-bit pairs over the first 32 columns of the buffers: this thread's kc
            // query columns are operand columns kc/2 * hf .. + kc/2 - 1
            if constexpr (HF == 2) {
                if (!warp_wait(BAR(LD_DONE), n & 1, P.status, ST_BWD_COMPUTE, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if constexpr (HF == 1) {
                tmem_st32(tbase + lane_off + bf * 64, pk);
                tmem_st32(tbase + lane_off + 128 + bf * 64, dk);
            } else {
                tmem_st16(tbase + lane_off + bf * 64 + 16 * hf, pk);
                tmem_st16(tbase + lane_off + 128 + bf * 64 + 16 * hf, dk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(PT_FULL(bf)));
        }
        // epilogue: dV, dK (x scale) for this key row; zero when no query sees it.  The
        // (part, 64-column half) slices q = part * (HD/64) + half leave as tiled stores
        // of 32 rows x 64 columns through 4 KB staging slices (rows past Tk are not
        // written): with HF = 1 each warp stores all of its rows' slices through two
        // alternating staging slices, with HF = 2 the two warps of a lane quarter split
        // them by q % 2, one staging slice each.
        const bool have = ok && ntiles > 0 && warp_wait(BAR(ACC_DONE), 0, P.status, ST_BWD_COMPUTE, &abort_flag);
        if (have) tc_fence_after();
        fence_proxy_async_smem();  // the staging slices reuse the Q ring the tensor core read
        // A packed sequence's last keys may share a 32-row slice with the next
        // sequence's first: such a slice goes out row by row (this sequence's rows
        // only).  Dense tensors end where the maps end, which clips the tiled store.
        const bool whole = !VL || j0 + wq * 32 + 32 <= sq.tk;
        if ((have || (ok && ntiles == 0)) && HF == 1) {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint32_t tcol = part == 0 ? tDV : tDK;
                const float mul = part == 0 ? 1.f : P.scale;
                uint32_t acc[HD / 32][32];
                if (have) {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) tmem_ld32(tcol + lane_off + c * 32, acc[c]);
                    tmem_ld_wait_only();
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) tmem_pin(acc[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[c][e] = 0u;
                }
                if (!whole) {
                    if (j < sq.tk) {
                        uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(part == 0 ? P.dv : P.dk) +
                                                              ((long long)sq.k0 + j) * P.Hkv * HD + (long long)kvh * HD);
#pragma unroll
                        for (int w4 = 0; w4 < HD / 8; ++w4) {
                            uint32_t q4[4];
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int col = w4 * 8 + 2 * t;
                                q4[t] = pack2<BF16>(__uint_as_float(acc[col >> 5][col & 31]) * mul,
                                                    __uint_as_float(acc[col >> 5][(col & 31) + 1]) * mul);
                            }
                            row[w4] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
                        }
                    }
                    continue;
                }
#pragma unroll
                for (int half = 0; half < HD / 64; ++half) {
                    const int q = part * (HD / 64) + half;
                    const uint32_t slice = sbase + C::kStgOff + warp * 8192 + (q & 1) * 4096;
                    // the slices alternate: this one's last store is the older of the
                    // two most recent groups
                    if (elect_one()) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    __syncwarp();
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        uint32_t w4[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int col = half * 64 + jj * 8 + 2 * t;  // element column
                            w4[t] = pack2<BF16>(__uint_as_float(acc[col >> 5][col & 31]) * mul,
                                                __uint_as_float(acc[col >> 5][(col & 31) + 1]) * mul);
                        }
                        st_shared_v4(slice + lane * 128 + ((jj ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (elect_one()) {
                        tile_store<PADH, HD>(part == 0 ? &tmDV : &tmDK, slice, kvh, half * 64,
                                             sq.k0 + j0 + wq * 32, sq.zb);
                        bulk_commit_group();
                    }
                }
            }
        }
        if ((have || (ok && ntiles == 0)) && HF == 2) {
            // each warp one slice: the (part, half) slices q with q % 2 == hf
            const uint32_t slice = sbase + C::kStgOff + warp * 4096;
#pragma unroll
            for (int q = hf; q < 2 * (HD / 64); q += 2) {
                const int part = q / (HD / 64), half = q % (HD / 64);
                const uint32_t tcol = (part == 0 ? tDV : tDK) + half * 64;
                const float mul = part == 0 ? 1.f : P.scale;
                uint32_t acc[2][32];
                if (have) {
                    tmem_ld32(tcol + lane_off, acc[0]);
                    tmem_ld32(tcol + lane_off + 32, acc[1]);
                    tmem_ld_wait_only();
                    tmem_pin(acc[0]);
                    tmem_pin(acc[1]);
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[c][e] = 0u;
                }
                if (!whole) {
                    if (j < sq.tk) {
                        uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(part == 0 ? P.dv : P.dk) +
                                                              ((long long)sq.k0 + j) * P.Hkv * HD + (long long)kvh * HD +
                                                              half * 64);
#pragma unroll
                        for (int w4 = 0; w4 < 8; ++w4) {
                            uint32_t q4[4];
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int col = w4 * 8 + 2 * t;
                                q4[t] = pack2<BF16>(__uint_as_float(acc[col >> 5][col & 31]) * mul,
                                                    __uint_as_float(acc[col >> 5][(col & 31) + 1]) * mul);
                            }
                            row[w4] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
                        }
                    }
                    continue;
                }
                // the slice's previous store has finished reading it
                if (elect_one()) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    uint32_t w4[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int col = jj * 8 + 2 * t;  // element column within the half
                        w4[t] = pack2<BF16>(__uint_as_float(acc[col >> 5][col & 31]) * mul,
                                            __uint_as_float(acc[col >> 5][(col & 31) + 1]) * mul);
                    }
                    st_shared_v4(slice + lane * 128 + ((jj ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_one()) {
                    tile_store<PADH, HD>(part == 0 ? &tmDV : &tmDK, slice, kvh, half * 64, sq.k0 + j0 + wq * 32,
                                         sq.zb);
                    bulk_commit_group();
                }
            }
        }
        if (elect_one()) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ===================================================================== dQ
template <int HD, bool OSTG = false>
struct QCfg {
    static constexpr int BQ = 128;  // query rows per item
    static constexpr int BK = 64;   // keys per inner tile
    static constexpr int kBoxes = HD / 64;
    // OSTG: the next item's O tile (for D = rowsum(dO*O)), and then D, land in the
    // epilogue staging between epilogues, which leaves room for a fourth K/V stage at
    // hd 128; otherwise O has a tile of its own.
    static constexpr int kStages = OSTG || HD != 128 ? 4 : 3;
    static constexpr int kQBytes = BQ * HD * 2;
    static constexpr int kKBytes = BK * HD * 2;  // one K (or V) tile
    static constexpr int kQOff = 0;
    static constexpr int kGOff = kQBytes;  // dO
    static constexpr int kKOff = (OSTG ? 2 : 3) * kQBytes;
    static constexpr int kVOff = kKOff + kStages * kKBytes;
    static constexpr int kBarOff = kVOff + kStages * kKBytes;
    static constexpr int kNumBars = 11 + 2 * kStages;
    // epilogue staging: one 32-row x 64-column slice (4 KB) per compute warp (8)
    static constexpr int kStgOff = (kBarOff + kNumBars * 8 + 16 + 1023) / 1024 * 1024;
    static constexpr int kOOff = OSTG ? kStgOff : 2 * kQBytes;  // O, then D of its rows
    static constexpr int kBytes = kStgOff + 8 * 4096;
    static constexpr int kLaunchBytes = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
    static_assert(!OSTG || kQBytes <= 8 * 4096, "the O tile fits in the staging slices");
};
// shared memory a dQ launch asks for (either layout)
template <int HD>
constexpr int dq_launch_bytes() {
    return QCfg<HD, false>::kLaunchBytes > QCfg<HD, true>::kLaunchBytes ? QCfg<HD, false>::kLaunchBytes
                                                                          : QCfg<HD, true>::kLaunchBytes;
}

// One dQ work item: 128 query rows of one (batch, head) and the key tiles they
// see.  Items are numbered longest first (every head's last query block first).
struct DqItem {
    int b, h, kvh, i0, kt0, ntiles;
    Seq sq;
};
template <int BQ, int BK, bool VL, bool RB = false>
__device__ __forceinline__ DqItem dq_item_at(const Params& P, int b, int h, int qb) {
    DqItem it;
    it.h = h;
    it.b = b;
    it.kvh = it.h / P.G;
    it.i0 = qb * BQ;
    it.sq = seq_of<VL>(P, it.b);
    int lo = 0, hi = 0;
    if (it.i0 < it.sq.tq) {  // (packed) items past a sequence's rows have no tiles
        const int ilast = min(it.i0 + BQ, it.sq.tq) - 1;
        key_range(P.wl, P.wr, it.sq.tk, it.i0 + P.q_offset, ilast + P.q_offset, &lo, &hi);
        if constexpr (RB) {  // packed fused-QKV rows: between the first row's sequence start and the last's end
            lo = max(lo, row_keys(P, it.i0, it.sq.tk).x);
            hi = max(lo, min(hi, row_keys(P, ilast, it.sq.tk).y));
        }
    }
    it.kt0 = lo / BK;
    it.ntiles = hi > lo ? (hi + BK - 1) / BK - it.kt0 : 0;
    return it;
}
// Packed batches of at most kVlCompact sequences: only the query blocks that hold rows
// of their own sequence are items.  Items run from the highest block index down; a
// level holds H items for every sequence that reaches it, sequences in order, heads
// innermost.  Lane b of a warp reads sequence b's block count, and a cursor walks the
// levels once, so each sequence of calls must have non-decreasing item numbers; every
// call is made by whole warps.  Otherwise items are numbered block-major over every
// (batch, head), longest first, and the cursor is unused.
struct DqCursor {
    int level;      // the block index the cursor is at
    int first;      // number of that level's first item
    unsigned seqs;  // the sequences that reach that level
};
template <int BQ>
__device__ __forceinline__ int dq_vl_blocks(const Params& P, int b) {
    return b < P.B ? (seq_of<true>(P, b).tq + BQ - 1) / BQ : 0;
}
// the item count; sets the cursor at the first level
template <int BQ, bool VL>
__device__ __forceinline__ int dq_items(const Params& P, DqCursor& c) {
    if (VL && P.B <= kVlCompact) {
        const int nb = dq_vl_blocks<BQ>(P, threadIdx.x & 31);
        c.level = (int)__reduce_max_sync(0xffffffffu, (unsigned)nb) - 1;
        c.first = 0;
        c.seqs = __ballot_sync(0xffffffffu, nb > 0 && nb > c.level);
        return (int)__reduce_add_sync(0xffffffffu, (unsigned)nb) * P.H;
    }
    return (P.Tq + BQ - 1) / BQ * P.H * P.B;
}
template <int BQ, int BK, bool VL, bool RB = false>
__device__ __forceinline__ DqItem dq_item(const Params& P, int w, DqCursor& c) {
    if (VL && P.B <= kVlCompact) {
        while (w >= c.first + __popc(c.seqs) * P.H && c.level > 0) {
            c.first += __popc(c.seqs) * P.H;
            --c.level;
            c.seqs = __ballot_sync(0xffffffffu, dq_vl_blocks<BQ>(P, threadIdx.x & 31) > c.level);
        }
        const int r = w - c.first, j = r / P.H;
        unsigned m = c.seqs;
        for (int t = 0; t < j && m; ++t) m &= m - 1;
        // (w is below the item count, so the sequence exists)
        return dq_item_at<BQ, BK, VL, RB>(P, m ? __ffs(m) - 1 : 0, r - j * P.H, c.level);
    }
    if constexpr (RB) {  // packed fused-QKV rows (one batch): blocks heaviest first
        if (P.item_order) return dq_item_at<BQ, BK, VL, RB>(P, 0, w % P.H, __ldg(P.item_order + w / P.H));
    }
    const int nqb = (P.Tq + BQ - 1) / BQ;
    const int hb = w % (P.H * P.B);
    return dq_item_at<BQ, BK, VL, RB>(P, hb / P.H, hb % P.H, nqb - 1 - w / (P.H * P.B));
}

// Persistent: one CTA per SM walks its items in snake order (snake_item).  The
// kernel also computes D = rowsum(dO*O) and LSE*log2(e) of its rows from the O
// and dO tiles it loads, uses them, and writes them into the workspace for the
// dK/dV pass (which therefore runs after this one).  The
// K/V ring and every barrier phase run on across items.  The next item's Q and dO
// are loaded into shared memory once the current ones are in TMEM, and copied
// into TMEM right after the current item's last dS, so its first S and dP run
// while the current item's epilogue reads dQ out.
template <bool BF16, int HD, int MODE>
__global__ void __launch_bounds__(kThreadsDQ, 1)
    bwd_dq_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                  const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmDQ) {
    // at hd 128 without a softcap O shares the epilogue staging and the K/V ring gets a
    // fourth stage (GQA prefill dQ 0.2007 -> 0.1884 ms); the softcap instantiations,
    // bound by their element work, measured slower that way (0.2314 -> 0.2335 ms)
    constexpr bool OSTG = HD == 128 && (MODE & 4) == 0;
    using C = QCfg<HD, OSTG>;
    constexpr int NS = C::kStages, BQ = C::BQ, BK = C::BK;
    // MODE & 3 as for dK/dV; MODE & 4: softcap; MODE & 8: a head size below HD (4-D maps)
    constexpr bool VL = (MODE & 3) == 1, BIAS = (MODE & 3) == 2, PADH = (MODE & 8) != 0;
    constexpr bool RB = (MODE & 64) != 0;  // packed fused-QKV rows: per-row sequence bounds
    static_assert(!RB || MODE == 64, "the row bounds are built for dense batches without other modes");
    static_assert(!(PADH && VL), "padded head sizes are built for dense batches only");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    __shared__ int abort_flag;
    // compute-warp epilogues whose staging slices have been read out (8 per item):
    // an O tile may land in the staging only after every epilogue before it
    __shared__ int stg_done;
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int QG_FULL = 0;   // Q, dO and O of an item in shared memory
    const int QG_EMPTY = 1;  // ... copied into TMEM (8 compute warps)
    const int QT_READY = 2;  // Q and dO of an item in TMEM (A operands; 8 warps)
    const int DQ_DONE = 3;   // the item's last dQ MMA completed
    const int DQ_EMPTY = 4;  // the epilogue has read dQ out of TMEM (8 warps)
    const int MMA_DONE = 5;
    auto ST_FULL = [&](int b) { return 6 + b; };  // S and dP of a tile (two issuers)
    auto DS_FULL = [&](int b) { return 8 + b; };  // dS of a tile (8 warps)
    auto KV_FULL = [&](int s) { return 10 + s; };
    auto KV_EMPTY = [&](int s) { return 10 + NS + s; };
    const int D_FULL = 10 + 2 * NS;  // D of an item's rows in shared memory (the Q/dO/O producer)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // every warp keeps its own cursors over the item sequence (one per monotone walk)
    DqCursor cur;
    const int nitems = dq_items<BQ, VL>(P, cur);
    DqCursor cur2 = cur;  // the compute warps' look-ahead walk

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            uint32_t count = 1;
            if (i == DS_FULL(0) || i == DS_FULL(1) || i == QT_READY || i == QG_EMPTY || i == DQ_EMPTY) count = 8;
            if (i == ST_FULL(0) || i == ST_FULL(1) || i == MMA_DONE) count = 2;  // two MMA issuers
            for (int s2 = 0; s2 < NS; ++s2)
                if (i == KV_EMPTY(s2)) count = 2;
            mbar_init(BAR(i), count);
        }
        abort_flag = 0;
        stg_done = 0;
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
    const uint32_t tDQ = tbase + 256;
    // Q and dO as 16-bit A operands in TMEM (row = lane, two elements per column):
    // every GEMM here then reads only K or V from shared memory
    const uint32_t tQ = tbase + 256 + HD, tG = tQ + HD / 2;

    if (warp >= 8) {
    regs_dec<kDqRegsAux>();
    if (warp == 11) {
        // ------------------------------- Q/dO/O producer and D (whole warp)
        // Loads the next item's tiles as soon as the current ones are in TMEM, then
        // forms D = rowsum(dO*O) of its 128 rows (lane l: rows l, l+32, l+64, l+96)
        // into the first 512 bytes of the O tile, and writes -D and -LSE*log2(e) of
        // every row into the workspace for the dK/dV pass (rows that see no key and
        // padding rows: D = 0, LSE = -inf).
        if (elect_one()) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmG);
            prefetch_tmap(&tmO);
        }
        auto stats = [&](const DqItem& it, int i2, float dval) {
            if (i2 >= P.tq_pad) return;
            const long long srow = ((long long)it.b * P.H + it.h) * P.tq_pad + i2;
            float nl2 = -INFINITY;
            if (i2 < it.sq.tq) {
                const float l = P.lse_in[((long long)it.b * P.H + it.h) * P.Tq + i2];
                nl2 = l == -INFINITY ? -INFINITY : -l * kLog2e;
            }
            P.ndelta[srow] = i2 < it.sq.tq ? -dval : 0.f;
            P.nlse2[srow] = nl2;
        };
        int qn = 0;         // Q/dO/O loads so far
        int prev_act = -1;  // position of the last item loaded
        for (int k_ = 0, w = snake_item(0); w < nitems; w = snake_item(++k_)) {
            const DqItem it = dq_item<BQ, BK, VL, RB>(P, w, cur);
            if (it.ntiles == 0) {
#pragma unroll
                for (int m = 0; m < BQ / 32; ++m) stats(it, it.i0 + m * 32 + lane, 0.f);
                continue;
            }
            if (qn > 0 && !warp_wait(BAR(QG_EMPTY), (qn - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag)) break;
            if constexpr (OSTG) {
                // O goes into the epilogue staging: the epilogues of every item before
                // the previous loaded one (for the first, before this one) must be out
                // of it.  The compute warps copy this item's Q/dO and read its D before
                // the previous item's epilogue, so no later epilogue can touch the
                // staging before D is read.
                const int need = 8 * (prev_act >= 0 ? prev_act : k_);
                if (!__all_sync(0xffffffffu, count_wait(&stg_done, need, P.status, ST_BWD_PRODUCER, &abort_flag)))
                    break;
            }
            if (elect_one()) mbar_expect_tx(BAR(QG_FULL), 3 * C::kQBytes);
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx) {
                if (elect_one())
                    tile_load<PADH, HD>(sbase + C::kQOff + bx * (BQ * 128), &tmQ, BAR(QG_FULL), it.h, bx,
                                        it.sq.q0 + it.i0, it.sq.zb);
                if (elect_one())
                    tile_load<PADH, HD>(sbase + C::kGOff + bx * (BQ * 128), &tmG, BAR(QG_FULL), it.h, bx,
                                        it.sq.q0 + it.i0, it.sq.zb);
                if (elect_one())
                    tile_load<PADH, HD>(sbase + C::kOOff + bx * (BQ * 128), &tmO, BAR(QG_FULL), it.h, bx,
                                        it.sq.q0 + it.i0, it.sq.zb);
            }
            ++qn;
            prev_act = k_;
            if (!warp_wait(BAR(QG_FULL), (qn - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag)) break;
            float dv[BQ / 32];
#pragma unroll
            for (int m = 0; m < BQ / 32; ++m) {
                const int rr = m * 32 + lane;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int half = 0; half < HD / 64; ++half) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const int off = half * (BQ * 128) + rr * 128 + ((ch ^ (rr & 7)) << 4);
                        const uint4 g4 = *reinterpret_cast<const uint4*>(smem + C::kGOff + off);
                        const uint4 o4 = *reinterpret_cast<const uint4*>(smem + C::kOOff + off);
                        a0 += dot2<BF16>(g4.x, o4.x) + dot2<BF16>(g4.y, o4.y);
                        a1 += dot2<BF16>(g4.z, o4.z) + dot2<BF16>(g4.w, o4.w);
                    }
                }
                dv[m] = a0 + a1;
            }
            __syncwarp();  // every lane has read its O rows
            float* d_smem = reinterpret_cast<float*>(smem + C::kOOff);
#pragma unroll
            for (int m = 0; m < BQ / 32; ++m) d_smem[m * 32 + lane] = dv[m];
            fence_proxy_async_smem();  // before the next TMA load overwrites it
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(D_FULL));
#pragma unroll
            for (int m = 0; m < BQ / 32; ++m) stats(it, it.i0 + m * 32 + lane, dv[m]);
        }
        if (qn > 0) mbar_wait(BAR(QG_FULL), (qn - 1) & 1, P.status, ST_TEARDOWN, nullptr);
    } else if (warp == 8) {
        // ------------------------------------------- K/V producer (whole warp)
        if (elect_one()) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
        bool ok = true;
        int g = 0;  // K/V tiles loaded so far
        for (int k_ = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++k_)) {
            const DqItem it = dq_item<BQ, BK, VL, RB>(P, w, cur);
            for (int n = 0; n < it.ntiles; ++n) {
                const int s = g % NS, use = g / NS;
                if (use > 0 && !warp_wait(BAR(KV_EMPTY(s)), (use - 1) & 1, P.status, ST_BWD_PRODUCER, &abort_flag)) {
                    ok = false;
                    break;
                }
                const int jt = (it.kt0 + n) * BK;
                if (elect_one()) mbar_expect_tx(BAR(KV_FULL(s)), 2 * C::kKBytes);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx) {
                    if (elect_one())
                        tile_load<PADH, HD>(sbase + C::kKOff + s * C::kKBytes + bx * (BK * 128), &tmK,
                                            BAR(KV_FULL(s)), it.kvh, bx, it.sq.k0 + jt, it.sq.zb);
                    if (elect_one())
                        tile_load<PADH, HD>(sbase + C::kVOff + s * C::kKBytes + bx * (BK * 128), &tmV,
                                            BAR(KV_FULL(s)), it.kvh, bx, it.sq.k0 + jt, it.sq.zb);
                }
                ++g;
            }
        }
        // every copy in flight lands before the CTA exits
        for (int n = max(0, g - NS); n < g; ++n)
            mbar_wait(BAR(KV_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
    } else if (warp == 9 || warp == 10) {
        // Two MMA issuers, so that one's barrier waits overlap the other's issue:
        // warp 9 issues S and dQ (the dS of tile n sits over S(n), so S(n+2) must
        // follow dQ(n) in one stream), warp 10 issues dP.  ST_FULL, KV_EMPTY and
        // MMA_DONE count both.  Tiles are numbered across items (gt): ring slot
        // gt % NS, S/dP buffer gt & 1.
        const bool issues_dp = warp == 10;
        constexpr uint32_t idS = idesc_f16(BF16, BQ, BK, false, false);
        constexpr uint32_t idAcc = idesc_f16(BF16, BQ, HD, false, true);
        auto wait_all = [&](int bar, uint32_t parity) -> bool {
            return warp_wait(BAR(bar), parity, P.status, ST_BWD_MMA, &abort_flag);
        };
        // S(t) = Q K_t^T (warp 5) or dP(t) = dO V_t^T (warp 6) into buffer t & 1
        auto issue_one = [&](int t) -> bool {
            const int s = t % NS, bf = t & 1;
            if (!wait_all(KV_FULL(s), (t / NS) & 1)) return false;
            tc_fence_after();
            const uint32_t src = sbase + (issues_dp ? C::kVOff : C::kKOff) + s * C::kKBytes;
            const uint64_t bdesc = sdesc_sw128(src, 16, 1024);
            const uint32_t d = tbase + (issues_dp ? 128 : 0) + bf * 64;
            const uint32_t a = issues_dp ? tG : tQ;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t boff = ((kk >> 2) * (BK * 128) + (kk & 3) * 32) >> 4;
                mma_ts_e(d, a + kk * 8, bdesc + boff, idS, kk > 0 ? 1u : 0u);
            }
            mma_commit_e(BAR(ST_FULL(bf)));
            return true;
        };
        bool ok = true;
        int gt = 0, act = 0;
        for (int k_ = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++k_)) {
            const DqItem it = dq_item<BQ, BK, VL, RB>(P, w, cur);
            if (it.ntiles == 0) continue;
            ok = wait_all(QT_READY, act & 1);
            if (ok) ok = issue_one(gt);
            if (ok && it.ntiles > 1) ok = issue_one(gt + 1);
            for (int n = 0; ok && n < it.ntiles; ++n) {
                const int t = gt + n, s = t % NS, bf = t & 1;
                // tile t's dS is written (and its S, dP read) once DS_FULL completes
                if (!wait_all(DS_FULL(bf), (t >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (!issues_dp) {
                    // the first dQ MMA overwrites the accumulator: the previous item's
                    // epilogue must have read it
                    if (n == 0 && act > 0 && !wait_all(DQ_EMPTY, (act - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kdesc = sdesc_sw128(sbase + C::kKOff + s * C::kKBytes, BK * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_ts_e(tDQ, tbase + bf * 64 + pcol(kk), kdesc + ((kk * 2048) >> 4), idAcc,
                                   (n > 0 || kk > 0) ? 1u : 0u);
                } else {
                    tc_fence_after();
                }
                mma_commit_e(BAR(KV_EMPTY(s)));
                if (n + 2 < it.ntiles) ok = issue_one(t + 2);
            }
            if (ok && !issues_dp) mma_commit_e(BAR(DQ_DONE));
            gt += it.ntiles;
            ++act;
        }
        mma_commit_e(BAR(MMA_DONE));
        mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
    }
    } else {
        regs_inc<kDqRegsCompute>();
        // ------------------- compute: warps w and w+4 share rows (TMEM lane quarter
        // w % 4, one query row per thread) and split each tile's 64 key columns (hf)
        const int wq = warp & 3, hf = warp >> 2;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        constexpr bool cap = (MODE & 4) != 0;
        const float cap_in = P.scale / fmaxf(P.softcap, 1e-30f);
        const uint64_t sl2_2 = f2_make(P.scale_log2, P.scale_log2), one2 = f2_make(1.f, 1.f);
        bool ok = true;
        int gt = 0, act = 0, qc = 0;  // tiles, active items and Q/dO copies so far
        int copied = -1;              // item whose Q and dO are in TMEM
        float d_copied = 0.f;         // D = rowsum(dO*O) of this thread's row of that item
        float l_copied = -INFINITY;   // its LSE, loaded with the copy (used at the item's start)
        auto load_lse = [&](const DqItem& it2) -> float {
            const int i2 = it2.i0 + r;
            return i2 < it2.sq.tq ? P.lse_in[((long long)it2.b * P.H + it2.h) * P.Tq + i2] : -INFINITY;
        };
        // copy this thread's row of Q (hf 0) or dO (hf 1), 128-byte-swizzled smem, into
        // TMEM; both halves also form D of the row from dO and O in shared memory
        // Copy this thread's row of Q (hf 0) or dO (hf 1), 128-byte-swizzled smem,
        // into TMEM; read the row's D that the producer warp formed.
        auto copy_q = [&](int w2) -> bool {
            if (!warp_wait(BAR(QG_FULL), qc & 1, P.status, ST_BWD_COMPUTE, &abort_flag)) return false;
            {
                const uint8_t* src = smem + (hf == 0 ? C::kQOff : C::kGOff);
#pragma unroll
                for (int half = 0; half < HD / 64; ++half) {
                    uint32_t wv[32];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(src + half * (BQ * 128) + r * 128 +
                                                                         ((ch ^ (r & 7)) << 4));
                        wv[4 * ch] = v4.x;
                        wv[4 * ch + 1] = v4.y;
                        wv[4 * ch + 2] = v4.z;
                        wv[4 * ch + 3] = v4.w;
                    }
                    tmem_st32((hf == 0 ? tQ : tG) + lane_off + half * 32, wv);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            // the MMA warps may start on this item now
            if (lane == 0) mbar_arrive(BAR(QT_READY));
            // issued here, consumed at the item's start: the latency hides behind
            // the current item's epilogue
            l_copied = load_lse(dq_item<BQ, BK, VL, RB>(P, w2, cur2));
            if (!warp_wait(BAR(D_FULL), qc & 1, P.status, ST_BWD_COMPUTE, &abort_flag)) return false;
            d_copied = reinterpret_cast<const float*>(smem + C::kOOff)[r];
            ++qc;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(QG_EMPTY));  // Q, dO, O and D in shared memory are free
            copied = w2;
            return true;
        };
        for (int k_ = 0, w = snake_item(0); w < nitems; w = snake_item(++k_)) {
            const DqItem it = dq_item<BQ, BK, VL, RB>(P, w, cur);
            const int i = it.i0 + r;
            const int p = i + P.q_offset;
            const int tq = it.sq.tq, tk = it.sq.tk;
            const bool row_ok = i < tq;
            const int ntiles = it.ntiles;
            int2 rk_own = make_int2(0, tk);  // packed fused-QKV rows: this row's sequence
            if constexpr (RB) rk_own = row_keys(P, max(min(i, tq - 1), 0), tk);
            float lse2 = INFINITY, Dd = 0.f;
            if (ntiles > 0 && copied != w) ok = copy_q(w);
            if (row_ok && ntiles > 0) {
                lse2 = l_copied == -INFINITY ? INFINITY : l_copied * kLog2e;
                Dd = d_copied;
            }
            const uint64_t nl2 = f2_make(-lse2, -lse2), nd2 = f2_make(-Dd, -Dd);
            for (int n = 0; ok && n < ntiles; ++n) {
                const int t = gt + n, bf = t & 1;
                const int jt = (it.kt0 + n) * BK;
                // this warp's 32 key columns: jt + 32 hf + [0, 32)
                const int jc = jt + 32 * hf;
                uint32_t mbits = 0xffffffffu;
                if (P.key_mask) {
                    const float* mrow = P.key_mask + (long long)it.b * P.mask_bstride;
                    const int j = jc + lane;
                    mbits = __ballot_sync(0xffffffffu, j < tk && mrow[j] > 0.5f);
                }
                int clo = 0, chi = min(32, tk - jc);
                if (P.wr >= 0) chi = min(chi, p + P.wr - jc + 1);
                if (P.wl >= 0) clo = max(clo, p - P.wl - jc);
                if constexpr (RB) {  // packed fused-QKV rows: this row's sequence
                    clo = max(clo, rk_own.x - jc);
                    chi = min(chi, rk_own.y - jc);
                }
                if (!row_ok) chi = 0;
                // the additive bias of the row's 32 keys, loaded before the wait for S (0 past
                // the keys)
                float bv[BIAS ? 32 : 1];
                if constexpr (BIAS) {
                    const float* brow = P.bias + (long long)it.b * P.bias_sb + (long long)it.h * P.bias_sh +
                                        (long long)(row_ok ? i : 0) * P.bias_sq;
                    if (P.bias_sk == 1 && jc + 32 <= tk && ((reinterpret_cast<uintptr_t>(brow + jc) & 15u) == 0)) {
                        const float4* r4 = reinterpret_cast<const float4*>(brow + jc);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 v4 = __ldg(r4 + e);
                            bv[4 * e] = v4.x;
                            bv[4 * e + 1] = v4.y;
                            bv[4 * e + 2] = v4.z;
                            bv[4 * e + 3] = v4.w;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) bv[e] = jc + e < tk ? __ldg(brow + (long long)(jc + e) * P.bias_sk) : 0.f;
                    }
                }
                if (!warp_wait(BAR(ST_FULL(bf)), (t >> 1) & 1, P.status, ST_BWD_COMPUTE, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[32], dp[32];
                tmem_ld32(tbase + lane_off + bf * 64 + 32 * hf, sv);
                tmem_ld32(tbase + lane_off + 128 + bf * 64 + 32 * hf, dp);
                tmem_ld_wait_only();
                tmem_pin(sv);
                tmem_pin(dp);
                // the bias joins the raw score here, or, with a softcap (which comes first),
                // the capped score inside the element loop
                if constexpr (BIAS && !cap) {
                    if (row_ok) {
                        const float inv = 1.f / P.scale;
#pragma unroll
                        for (int e = 0; e < 32; ++e) sv[e] = __float_as_uint(fmaf(bv[e], inv, __uint_as_float(sv[e])));
                    }
                }
                uint32_t dsk[16];
                // with a softcap, the polynomial serves the tile unless a raw score of the
                // row lies outside its range (checked before masking)
                bool poly = false, shorter = false;
                if (cap) {
                    float amax = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 32; cc += 2)
                        amax = max3f(amax, fabsf(__uint_as_float(sv[cc])), fabsf(__uint_as_float(sv[cc + 1])));
                    poly = __all_sync(0xffffffffu, amax <= cap_poly(P.scale, P.softcap).r_max);
                    shorter = __all_sync(0xffffffffu, amax <= cap_short(P.scale, P.softcap).r_max);
                }
                // invisible pairs become -inf scores first: one copy of the element loop
                const bool full = row_ok && !P.key_mask && clo <= 0 && chi >= 32;
                if (!__all_sync(0xffffffffu, full)) {
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc)
                        sv[cc] = (cc >= clo && cc < chi && ((mbits >> cc) & 1u)) ? sv[cc] : 0xff800000u;
                    poly = poly && cap_poly(P.scale, P.softcap).inf_ok;
                    shorter = shorter && cap_short(P.scale, P.softcap).inf_ok;
                }
                // Mode 0: no softcap; 1: softcap by the polynomial; 2: by tanh_accurate; 3: by
                // the short polynomial.  Pairs of columns go through the f32x2 unit together.
                auto elems = [&](auto modec) {
                    constexpr int kMode = decltype(modec)::value;
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float s0 = __uint_as_float(sv[c]), s1 = __uint_as_float(sv[c + 1]);
                        const uint64_t dp2 = f2_make(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1]));
                        float x0, x1;
                        uint64_t dcap = one2;
                        // the bias (with a softcap) in log2 units, added after the cap
                        float b0 = 0.f, b1 = 0.f;
                        if constexpr (BIAS && cap) {
                            b0 = bv[c] * kLog2e;
                            b1 = bv[c + 1] * kLog2e;
                        }
                        if constexpr (kMode == 2) {
                            // softcap*tanh(-inf) would be finite: keep a masked score at -inf
                            const float t0 = tanh_accurate(s0 * cap_in), t1 = tanh_accurate(s1 * cap_in);
                            x0 = s0 == -INFINITY ? -INFINITY : fmaf(P.softcap * kLog2e, t0, b0 - lse2);
                            x1 = s1 == -INFINITY ? -INFINITY : fmaf(P.softcap * kLog2e, t1, b1 - lse2);
                            dcap = f2_make(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
                        } else {
                            uint64_t g = f2_make(s0, s1);
                            if constexpr (kMode == 1) {
                                uint64_t uu;
                                const CapPoly cp = cap_poly(P.scale, P.softcap);
                                g = cap_g(cp, g, uu);
                                // 1 - tanh^2; a masked score gives g = -inf and -inf here, with P = 0
                                float d0, d1;
                                f2_split(f2_fma(f2_mul(g, g), cp.nc2, one2), d0, d1);
                                dcap = f2_make(fmaxf(d0, 0.f), fmaxf(d1, 0.f));
                            } else if constexpr (kMode == 3) {
                                // the short polynomial (every raw score of the tile within its
                                // range); a masked score gives g = -inf as above
                                g = cap_g_short(cap_short(P.scale, P.softcap), g);
                                float d0, d1;
                                f2_split(f2_fma(f2_mul(g, g), cap_poly(P.scale, P.softcap).nc2, one2), d0, d1);
                                dcap = f2_make(fmaxf(d0, 0.f), fmaxf(d1, 0.f));
                            }
                            if constexpr (BIAS && cap) f2_split(f2_fma(g, sl2_2, f2_add(nl2, f2_make(b0, b1))), x0, x1);
                            else f2_split(f2_fma(g, sl2_2, nl2), x0, x1);
                        }
                        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                        uint64_t ds = f2_mul(f2_make(p0, p1), f2_add(dp2, nd2));
                        if constexpr (kMode != 0) ds = f2_mul(ds, dcap);
                        float q0, q1;
                        f2_split(ds, q0, q1);
                        dsk[c >> 1] = pack2<BF16>(q0, q1);
                    }
                };
                if (!cap) elems(std::integral_constant<int, 0>());
                else if (shorter) elems(std::integral_constant<int, 3>());
                else if (poly) elems(std::integral_constant<int, 1>());
                else elems(std::integral_constant<int, 2>());
                // packed into the first 16 of the 32 columns this warp read (the partner
                // warp may still be loading the other 32)
                tmem_st16(tbase + lane_off + bf * 64 + 32 * hf, dsk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(DS_FULL(bf)));
            }
            if (!ok) break;
            // every S and dP of this item completed (their results were read above):
            // put the next active item's Q and dO into TMEM before this epilogue
            for (int k2 = k_ + 1, w2 = snake_item(k2); ntiles > 0 && w2 < nitems; w2 = snake_item(++k2)) {
                if (dq_item<BQ, BK, VL, RB>(P, w2, cur2).ntiles == 0) continue;
                ok = copy_q(w2);
                break;
            }
            if (!ok) break;
            // epilogue: dQ (x scale) of this row, zero when it sees no key
            const bool have = ntiles > 0 && warp_wait(BAR(DQ_DONE), act & 1, P.status, ST_BWD_COMPUTE, &abort_flag);
            if (ntiles > 0) {
                if (!have) {
                    ok = false;
                    break;
                }
                ++act;
                tc_fence_after();
            }
            // columns of dQ this warp writes: 64 * hf + [0, 64) (hd 128); the whole row
            // by hf 0 (hd 64)
            constexpr int kCols = 64;
            const bool writes = HD == 128 || hf == 0;
            const int c0 = HD == 128 ? 64 * hf : 0;
            uint32_t packed[kCols / 2];
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c) {
                uint32_t acc[32];
                if (have && writes) {
                    tmem_ld32(tDQ + lane_off + c0 + c * 32, acc);
                    tmem_ld_wait(acc);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    packed[c * 16 + e] = pack2<BF16>(__uint_as_float(acc[2 * e]) * P.scale,
                                                     __uint_as_float(acc[2 * e + 1]) * P.scale);
            }
            if (have) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(DQ_EMPTY));
            }
            // A packed sequence's last rows may share a 32-row slice with the next
            // sequence's first (or lie past its end): such a slice goes out row by row,
            // this sequence's rows only.  Dense tensors end where the map ends.
            const bool whole = !VL || it.i0 + wq * 32 + 32 <= tq;
            if (writes && !whole && row_ok) {
                uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(P.dq) +
                                                      ((long long)it.sq.q0 + i) * P.H * HD + (long long)it.h * HD + c0);
#pragma unroll
                for (int w4 = 0; w4 < kCols / 8; ++w4)
                    row[w4] = make_uint4(packed[4 * w4], packed[4 * w4 + 1], packed[4 * w4 + 2], packed[4 * w4 + 3]);
            }
            // this warp's 32 rows x 64 columns leave through its staging slice
            if (writes && whole) {
                const uint32_t slice = sbase + C::kStgOff + warp * 4096;
                if (elect_one()) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(slice + lane * 128 + ((j ^ (lane & 7)) << 4), packed[4 * j], packed[4 * j + 1],
                                 packed[4 * j + 2], packed[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_one()) {
                    tile_store<PADH, HD>(&tmDQ, slice, it.h, c0, it.sq.q0 + it.i0 + wq * 32, it.sq.zb);
                    bulk_commit_group();
                }
            }
            if constexpr (OSTG) {
                // the staging may take the next O tile once this warp's store has read its slice
                if (elect_one()) bulk_wait_read_all();
                __syncwarp();
                if (lane == 0) atomicAdd(&stg_done, 1);
            }
            gt += ntiles;
        }
        if (elect_one()) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// Pass 4 (dQ) forms D and LSE*log2(e) itself and writes them (negated) into the
// workspace, so with pass 4 requested pass 1 is not run separately, and dQ goes
// before dK/dV, which reads them.
template <bool BF16, int HD>
cudaError_t bwd_typed(const Params& p, const BwdMaps& m, int phases, cudaStream_t s) {
    cudaError_t e;
    if ((phases & 1) && !(phases & 4)) {
        e = launch_bwd_preprocess(p, BF16 ? 2 : 1, s);
        if (e != cudaSuccess) return e;
    }
    if (phases & 4) {
        // a head size below HD (dense batches without a bias only) runs the padded instantiations
        const bool c = p.softcap > 0.f;
        auto k = p.hd != HD ? (c ? bwd_dq_kernel<BF16, HD, 12> : bwd_dq_kernel<BF16, HD, 8>)
                 : p.cu_q   ? (c ? bwd_dq_kernel<BF16, HD, 5> : bwd_dq_kernel<BF16, HD, 1>)
                 : p.row_bounds ? bwd_dq_kernel<BF16, HD, 64>
                 : p.bias   ? (c ? bwd_dq_kernel<BF16, HD, 6> : bwd_dq_kernel<BF16, HD, 2>)
                            : (c ? bwd_dq_kernel<BF16, HD, 4> : bwd_dq_kernel<BF16, HD, 0>);
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_launch_bytes<HD>());
        if (e != cudaSuccess) return e;
        int dev = 0, nsm = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        // persistent: one CTA per SM (one fits); each walks its items in snake order
        const long long items = (long long)((p.Tq + 127) / 128) * p.H * p.B;
        const unsigned grid = (unsigned)(items < nsm ? items : nsm);
        k<<<grid, kThreadsDQ, dq_launch_bytes<HD>(), s>>>(p, m.q, m.k64, m.v64, m.dout, m.o, m.dq32);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (phases & 2) {
        const bool c = p.softcap > 0.f;
        auto k = p.hd != HD ? (c ? bwd_dkdv_kernel<BF16, HD, 12> : bwd_dkdv_kernel<BF16, HD, 8>)
                 : p.cu_q   ? (c ? bwd_dkdv_kernel<BF16, HD, 5> : bwd_dkdv_kernel<BF16, HD, 1>)
                 : p.row_bounds ? bwd_dkdv_kernel<BF16, HD, 64>
                 : p.bias   ? (c ? bwd_dkdv_kernel<BF16, HD, 6> : bwd_dkdv_kernel<BF16, HD, 2>)
                            : (c ? bwd_dkdv_kernel<BF16, HD, 4> : bwd_dkdv_kernel<BF16, HD, 0>);
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, KVCfg<HD>::kLaunchBytes);
        if (e != cudaSuccess) return e;
        const unsigned grid = (unsigned)((p.Tk + 127) / 128) * p.Hkv * p.B;
        // about 32 MB of Q and dO per chunk of (batch, KV head) pairs
        Params pc = p;
        const long long per = 2LL * p.G * p.Tq * p.hd * 2;
        // (packed sequences differ in length: their key blocks keep one global order)
        pc.kv_chunk = p.cu_q ? 0 : (int)std::max(1LL, std::min<long long>(p.Hkv * p.B, (32LL << 20) / std::max(per, 1LL)));
        const int threads = c ? dkdv_threads(4) : dkdv_threads(0);
        k<<<grid, threads, KVCfg<HD>::kLaunchBytes, s>>>(pc, m.q64, m.k, m.v, m.dout64, m.dk32, m.dv32);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

}  // namespace attn
