// fwd_tc.cuh -- prefill forward on the 5th-generation tensor cores (sm_103a).
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

#pragma once

#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;      // query rows per tile (two tiles per CTA)
constexpr int BN = 128;      // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleHi = 8.0f;   // log2 units: the row max may reach 2^8 times the reference
constexpr float kRescaleLo = -2.0f;  // a row's first visible tile may put its max at >= 2^-2

struct TileInfo {
    int t0, ntiles;
};

// key tiles the query tile at rows i0 .. of a sequence of tq queries and tk keys sees,
// within the span of keys the key mask keeps (span.y <= span.x: none)
__device__ __forceinline__ TileInfo tile_range(const Params& P, int i0, int tq, int tk, int2 span) {
    const int p0 = i0 + P.q_offset;
    const int p1 = min(i0 + BM, tq) - 1 + P.q_offset;
    int lo, hi;
    key_range(P.wl, P.wr, tk, p0, p1, &lo, &hi);
    lo = max(lo, span.x);
    hi = min(hi, span.y);
    TileInfo t;
    t.t0 = lo / BN;
    t.ntiles = hi > lo ? (hi + BN - 1) / BN - t.t0 : 0;
    return t;
}

// ------------------------------------------------------------------------
// Persistent: one CTA per SM walks work items in snake order (items c, 2g-1-c,
// 2g+c, ... for CTA c of g), so that the heavy first items and the light last
// ones even out across the CTAs.  An item is two query tiles (256 rows of one
// head) sharing every K/V tile, with one softmax warpgroup per tile, so the
// tensor core works on one tile's
// P.V and next S while the other warpgroup runs its softmax (ping-pong).  The
// K/V ring and every barrier phase run on across items: the next item's Q tile
// loads once the current item's last S of that tile completed, and its first
// P.V waits only for the epilogue to have read O out of TMEM, so item
// boundaries cost little more than a ring step.
//   warps 0-3  softmax of tile A (rows i0 .. i0+127)
//   warps 4-7  softmax of tile B (rows i0+128 .. i0+255)
//   warp 8     TMA producer     warp 9  TMEM owner + MMA issuer of tile A
//   warp 10    MMA issuer of tile B                                 (11 idle)
// Registers: launched at 168 per thread (384 threads = 64512); the producer
// warpgroup gives its share to the softmax warpgroups with setmaxnreg
// (2*128*216 + 128*72 = 64512, never more than the launch total).
// TMEM: S_A 0, S_B 128, O_A 256, O_B 256+hd (512 columns).  Each tile has a
// single S buffer; S_u(n) is issued after P_u(n-1) V(n-1), so a completed
// S_u(n) also means O_u is stable for a rescale.
constexpr int kThreads2 = 384;
constexpr int kRegsSoftmax = 216, kRegsProducer = 72;
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
    static constexpr int kNumBars = 15 + 4 * kStages;
    // epilogue staging: one 32-row x 64-column slice (4 KB) per softmax warp
    static constexpr int kStgOff = (kBarOff + kNumBars * 8 + 16 + 1023) / 1024 * 1024;
    static constexpr int kStgBytes = 8 * 32 * 128;
    static constexpr int kBytes = kStgOff + kStgBytes;
    static constexpr int kLaunchBytes = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

// One work item: 256 query rows (tiles A and B) of one (batch, head), and the
// key tiles each tile sees.  Items are numbered longest first: every head's last
// (causally heaviest) query block comes before any head's next one.
struct FwdItem {
    int b, h, kvh, i0;
    Seq sq;
    bool hasB;
    TileInfo tu[2];
    int t0, ntiles;  // union key-tile range of the two tiles
};

// The item of query block cq (rows 256*cq ..) of head h in sequence b; an item
// that is not valid has no rows.
// kspan: the key-mask spans of the batches (shared memory), or NULL for none
template <bool VL, bool RB = false>
__device__ __forceinline__ FwdItem make_item(const Params& P, int b, int h, int cq, bool valid, const int2* kspan) {
    FwdItem it;
    it.h = h;
    it.b = b;
    it.kvh = it.h / P.G;
    it.i0 = cq * 2 * BM;
    it.sq = seq_of<VL>(P, it.b);
    if (!valid) it.sq.tq = 0;
    it.hasB = it.i0 + BM < it.sq.tq;
    const int2 span = kspan ? kspan[b] : make_int2(0, it.sq.tk);
    // packed fused-QKV rows: a tile's keys lie between its first row's sequence start
    // and its last row's sequence end
    auto span_of = [&](int i0) -> int2 {
        if constexpr (!RB) {
            return span;
        } else {
            const int ilast = min(i0 + BM, it.sq.tq) - 1;
            return make_int2(max(span.x, row_keys(P, i0, it.sq.tk).x), min(span.y, row_keys(P, ilast, it.sq.tk).y));
        }
    };
    it.tu[0] = it.i0 < it.sq.tq ? tile_range(P, it.i0, it.sq.tq, it.sq.tk, span_of(it.i0)) : TileInfo{0, 0};
    it.tu[1] = it.hasB ? tile_range(P, it.i0 + BM, it.sq.tq, it.sq.tk, span_of(it.i0 + BM)) : TileInfo{0, 0};
    int t0 = it.tu[0].t0, t1 = it.tu[0].t0 + it.tu[0].ntiles;
    if (it.tu[1].ntiles > 0) {
        if (it.tu[0].ntiles == 0) {
            t0 = it.tu[1].t0;
            t1 = it.tu[1].t0 + it.tu[1].ntiles;
        } else {
            t0 = min(t0, it.tu[1].t0);
            t1 = max(t1, it.tu[1].t0 + it.tu[1].ntiles);
        }
    }
    it.t0 = t0;
    it.ntiles = t1 > t0 ? t1 - t0 : 0;
    return it;
}
__device__ __forceinline__ int fwd_items(const Params& P) { return (P.Tq + 2 * BM - 1) / (2 * BM) * P.H * P.B; }

// Packed sequences, at most 32 of them (kVlCompact): only the query blocks that
// hold rows of their own sequence become items, so no CTA is dealt empty items
// in place of work.  Items run from the highest block index down (the heaviest
// under a causal mask first); a level holds H items for every sequence that
// reaches it, sequences in order, heads innermost.  Lane b of a warp reads
// sequence b's block count, and a cursor walks the levels once per CTA, as the
// CTA's item numbers only grow.  Every call is made by whole warps.  More
// sequences keep the plain numbering (a sequence's surplus items have no rows).
struct VlCursor {
    int level;      // the block index the cursor is at
    int first;      // number of that level's first item
    unsigned seqs;  // the sequences that reach that level
};
// query blocks of 2*BM rows of sequence b (0 past the batch)
__device__ __forceinline__ int vl_blocks(const Params& P, int b) {
    return b < P.B ? (seq_of<true>(P, b).tq + 2 * BM - 1) / (2 * BM) : 0;
}
__device__ __forceinline__ int vl_init(const Params& P, VlCursor& c, int lane) {
    const int nb = vl_blocks(P, lane);
    c.level = (int)__reduce_max_sync(0xffffffffu, (unsigned)nb) - 1;
    c.first = 0;
    c.seqs = __ballot_sync(0xffffffffu, nb > 0 && nb > c.level);
    return (int)__reduce_add_sync(0xffffffffu, (unsigned)nb) * P.H;
}
// item w (not below any earlier call's w, and below the item count)
__device__ __forceinline__ FwdItem vl_item(const Params& P, VlCursor& c, int w) {
    while (w >= c.first + __popc(c.seqs) * P.H && c.level > 0) {
        c.first += __popc(c.seqs) * P.H;
        --c.level;
        c.seqs = __ballot_sync(0xffffffffu, vl_blocks(P, threadIdx.x & 31) > c.level);
    }
    const int r = w - c.first, j = r / P.H;
    unsigned m = c.seqs;
    for (int t = 0; t < j && m; ++t) m &= m - 1;
    const bool valid = r >= 0 && r < __popc(c.seqs) * P.H && m != 0u;
    return make_item<true>(P, valid ? __ffs(m) - 1 : 0, valid ? r - j * P.H : 0, c.level, valid, nullptr);
}

// The additive bias of row i over the key tile j0 .. j0+127 (0 past the keys), loaded
// into registers before the tile's scores are needed, so that the loads' latency runs
// under the waits for S and for the other tile's softmax.  Rows of 16-byte-aligned
// contiguous bias load as float4.
__device__ __forceinline__ void load_bias_row(const Params& P, int b, int h, int i, int j0, int tk,
                                              float (&bv)[128]) {
    const float* row = P.bias + (long long)b * P.bias_sb + (long long)h * P.bias_sh + (long long)i * P.bias_sq;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int jc = j0 + 32 * c;
        if (P.bias_sk == 1 && jc + 32 <= tk && ((reinterpret_cast<uintptr_t>(row + jc) & 15u) == 0)) {
            const float4* r4 = reinterpret_cast<const float4*>(row + jc);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 v = __ldg(r4 + e);
                bv[32 * c + 4 * e] = v.x;
                bv[32 * c + 4 * e + 1] = v.y;
                bv[32 * c + 4 * e + 2] = v.z;
                bv[32 * c + 4 * e + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                bv[32 * c + e] = jc + e < tk ? __ldg(row + (long long)(jc + e) * P.bias_sk) : 0.f;
        }
    }
}

// KORD: dense key-masked batches with their spans in kspan and kord the batches by
// kept span, longest first.  Without a window every query block of a batch sees
// the same key tiles, so a batch's items run together, the longest spans first;
// otherwise each level of query blocks takes its batches in that order.
template <bool VL, bool KORD = false, bool RB = false>
__device__ __forceinline__ FwdItem fwd_item(const Params& P, int w, VlCursor& c, const int2* kspan,
                                            const unsigned char* kord = nullptr) {
    if constexpr (VL) {
        if (P.B <= kVlCompact) return vl_item(P, c, w);
    }
    const int ncq = (P.Tq + 2 * BM - 1) / (2 * BM);
    if constexpr (RB) {  // packed fused-QKV rows (one batch): blocks heaviest first
        if (P.item_order) return make_item<VL, RB>(P, 0, w % P.H, __ldg(P.item_order + w / P.H), true, kspan);
    }
    if constexpr (KORD) {
        if (P.wl < 0 && P.wr < 0) {
            const int per = P.H * ncq, rem = w % per;
            return make_item<VL, RB>(P, kord[w / per], rem % P.H, rem / P.H, true, kspan);
        }
        const int hb = w % (P.H * P.B);
        return make_item<VL, RB>(P, kord[hb / P.H], hb % P.H, ncq - 1 - w / (P.H * P.B), true, kspan);
    }
    const int hb = w % (P.H * P.B);
    return make_item<VL, RB>(P, hb / P.H, hb % P.H, ncq - 1 - w / (P.H * P.B), true, kspan);
}

// MODE & 3 -- 0: dense; 1: packed variable-length sequences (cu_seqlens); 2: dense with
// an additive score bias; MODE & 4: softcap; MODE & 8: a head size below HD (96 in a
// 128 kernel, 32 in a 64 kernel) read and written through 4-D maps whose boxes reach
// past the head (the extra columns load as zeros, add nothing to q.k or P.V, and are
// never stored); MODE & 16: rotary embedding of the query tiles in shared memory
// (dense batches): the softmax warps of a tile turn their rows' pairs (x[c],
// x[c + hd/2]) by the angles of P.rope_tab once the tile lands, and the MMA warp
// waits for that (Q_ROT) instead of the load.  Each instantiation carries only its
// own bookkeeping.  MODE & 32: dense key-masked batches (at most kMaskSpanMax of
// them), the items numbered by the batches' kept key spans, longest first.  MODE 64:
// packed fused-QKV rows of one batch, each query row limited to its own sequence's
// keys (P.row_bounds) inside the window.
template <bool BF16, int HD, int MODE>
__global__ void __launch_bounds__(kThreads2, 1)
    fwd_tc2_kernel(const Params P, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO) {
    constexpr bool VL = (MODE & 3) == 1, BIAS = (MODE & 3) == 2, PADH = (MODE & 8) != 0, ROPE = (MODE & 16) != 0;
    constexpr bool RB = (MODE & 64) != 0;  // packed fused-QKV rows: per-row sequence bounds
    static_assert(!RB || MODE == 64, "the row bounds are built for dense batches without other modes");
    constexpr bool KORD = (MODE & 32) != 0;
    static_assert(!(KORD && (MODE & 31) != 0), "the span order is built for plain dense key-masked batches");
    static_assert(!(PADH && VL), "padded head sizes are built for dense batches only");
    static_assert(!(ROPE && (VL || BIAS || PADH)), "the fused rotation is built for dense batches at hd 64 / 128");
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
    auto Q_FULL = [&](int u) { return u; };
    auto Q_EMPTY = [&](int u) { return 2 + u; };  // the item's last S of tile u completed
    auto K_FULL = [&](int s) { return 4 + s; };
    auto K_EMPTY = [&](int s) { return 4 + NS + s; };
    auto V_FULL = [&](int s) { return 4 + 2 * NS + s; };
    auto V_EMPTY = [&](int s) { return 4 + 3 * NS + s; };
    auto S_FULL = [&](int u) { return 4 + 4 * NS + u; };
    auto P_FULL = [&](int u) { return 6 + 4 * NS + u; };
    auto O_DONE = [&](int u) { return 8 + 4 * NS + u; };   // the item's last P.V of tile u completed
    auto O_EMPTY = [&](int u) { return 10 + 4 * NS + u; };  // the epilogue has read O_u out of TMEM
    const int MMA_DONE = 12 + 4 * NS;
    auto Q_ROT = [&](int u) { return 13 + 4 * NS + u; };  // Q tile u rotated in shared memory (4 warps)
    // softmaxes finished by tile u, counted per warp (exact counts: a tile with no work
    // in an item lets the other run several softmaxes ahead, which mbarrier parity
    // could not tell apart)
    __shared__ int done_count[2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Key-mask spans per batch (dense batches of at most kMaskSpanMax): key tiles a
    // mask removes entirely at the ends of a row are never loaded or multiplied.  Each
    // warp scans the batches w, w + 12, ...; the spans are read after the block-wide
    // barrier below.
    // (KORD: the batch order in the 64 bytes past the spans)
    __shared__ int2 kspan_s[kMaskSpanMax + (KORD ? kMaskSpanMax / 8 : 0)];
    unsigned char* kord_s = reinterpret_cast<unsigned char*>(kspan_s + kMaskSpanMax);
    const int2* kspan = (!VL && P.key_mask && P.B <= kMaskSpanMax) ? kspan_s : nullptr;
    if (kspan)
        for (int b = warp; b < P.B; b += kThreads2 / 32) {
            const int2 sp = mask_span(P, b, P.Tk);
            if (lane == 0) kspan_s[b] = sp;
        }
    VlCursor vcur = {};
    int nitems = fwd_items(P);
    if constexpr (VL) {
        if (P.B <= kVlCompact) nitems = vl_init(P, vcur, lane);
    }
    // every role walks the same item sequence; a tile u is active in an item when
    // it has rows and sees at least one key tile
    // (tile u is a run-time value: select, so that the item stays in registers)
    auto active = [&](const FwdItem& it, int u) { return (u == 0 ? it.tu[0].ntiles : it.tu[1].ntiles) > 0; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            uint32_t count = 1;
            if (i == P_FULL(0) || i == P_FULL(1) || i == O_EMPTY(0) || i == O_EMPTY(1) || i == Q_ROT(0) ||
                i == Q_ROT(1))
                count = 4;
            // stage releases and the teardown barrier: one arrival per MMA issuer
            for (int s2 = 0; s2 < NS; ++s2)
                if (i == K_EMPTY(s2) || i == V_EMPTY(s2)) count = 2;
            if (i == MMA_DONE) count = 2;
            mbar_init(BAR(i), count);
        }
        abort_flag = 0;
        done_count[0] = done_count[1] = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (KORD) {
        // rank the batches by kept span, longest first (ties by index)
        if ((int)threadIdx.x < P.B) {
            const int b = threadIdx.x, len = kspan_s[b].y - kspan_s[b].x;
            int rank = 0;
            for (int b2 = 0; b2 < P.B; ++b2) {
                const int l2 = kspan_s[b2].y - kspan_s[b2].x;
                rank += (l2 > len || (l2 == len && b2 < b)) ? 1 : 0;
            }
            kord_s[rank] = (unsigned char)b;
        }
        __syncthreads();
    }
    const uint32_t tbase = *tmem_slot;
    if (warp >= 8) {
        regs_dec<kRegsProducer>();
        // The producer and the MMA issuers run their loops as whole warps and issue
        // each TMA copy, MMA and commit from one elected lane.
        if (warp == 8) {
            if (elect_one()) {
                prefetch_tmap(&tmQ);
                prefetch_tmap(&tmK);
                prefetch_tmap(&tmV);
            }
            bool ok = true;
            int gk = 0, gv = 0;   // K and V tiles loaded so far (ring positions)
            int qn[2] = {0, 0};   // Q tiles loaded so far, per tile slot
            for (int kw = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++kw)) {
                const FwdItem it = fwd_item<VL, KORD, RB>(P, w, vcur, kspan, kord_s);
                if (it.ntiles == 0) continue;
                for (int u = 0; ok && u < 2; ++u) {
                    if (!active(it, u)) continue;
                    // the slot is free once the previous item's last S of this tile completed
                    if (qn[u] > 0 && !warp_wait(BAR(Q_EMPTY(u)), (qn[u] - 1) & 1, P.status, ST_FWD_PRODUCER,
                                                &abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) mbar_expect_tx(BAR(Q_FULL(u)), C::kQBytes);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        if (elect_one())
                            tile_load<PADH, HD>(sbase + C::kQOff + u * C::kQBytes + bx * (BM * 128), &tmQ,
                                                BAR(Q_FULL(u)), it.h, bx, it.sq.q0 + it.i0 + u * BM, it.sq.zb);
                    ++qn[u];
                }
                for (int n = 0; ok && n < it.ntiles; ++n) {
                    const int s = gk % NS, use = gk / NS;
                    const int j0 = (it.t0 + n) * BN;
                    if (use > 0 && !warp_wait(BAR(K_EMPTY(s)), (use - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) mbar_expect_tx(BAR(K_FULL(s)), C::kKVBytes);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        if (elect_one())
                            tile_load<PADH, HD>(sbase + C::kKOff + s * C::kKVBytes + bx * (BN * 128), &tmK,
                                                BAR(K_FULL(s)), it.kvh, bx, it.sq.k0 + j0, it.sq.zb);
                    ++gk;
                    if (use > 0 && !warp_wait(BAR(V_EMPTY(s)), (use - 1) & 1, P.status, ST_FWD_PRODUCER, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) mbar_expect_tx(BAR(V_FULL(s)), C::kKVBytes);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        if (elect_one())
                            tile_load<PADH, HD>(sbase + C::kVOff + s * C::kKVBytes + bx * (BN * 128), &tmV,
                                                BAR(V_FULL(s)), it.kvh, bx, it.sq.k0 + j0, it.sq.zb);
                    ++gv;
                }
            }
            // every copy in flight lands before the CTA exits
            for (int u = 0; u < 2; ++u)
                if (qn[u] > 0) mbar_wait(BAR(Q_FULL(u)), (qn[u] - 1) & 1, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, gk - NS); n < gk; ++n)
                mbar_wait(BAR(K_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
            for (int n = max(0, gv - NS); n < gv; ++n)
                mbar_wait(BAR(V_FULL(n % NS)), (n / NS) & 1, P.status, ST_TEARDOWN, nullptr);
        } else if (warp == 9 || warp == 10) {
            // Two MMA issuers, one per query tile (warp 9: A, warp 10: B), so that one
            // tile's barrier waits overlap the other tile's MMA issue.  Each runs its own
            // in-order chain over the same items; both commit the K/V stage releases of
            // every tile (those barriers count one arrival per issuer).
            const int u = warp - 9;
            constexpr uint32_t idS = idesc_f16(BF16, BM, BN, false, false);
            constexpr uint32_t idPV = idesc_f16(BF16, BM, HD, false, true);
            auto wait_all = [&](int bar, uint32_t parity) -> bool {
                return warp_wait(BAR(bar), parity, P.status, ST_FWD_MMA, &abort_flag);
            };
            const uint64_t qdesc = sdesc_sw128(sbase + C::kQOff + u * C::kQBytes, 16, 1024);
            const uint32_t tS = tbase + u * 128, tO = tbase + 256 + u * HD;
            bool ok = true;
            int g = 0;    // ring position of the item's first tile
            int pc = 0;   // P_FULL(u) phases consumed
            int act = 0;  // items in which this tile was active so far
            for (int kw = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++kw)) {
                const FwdItem it = fwd_item<VL, KORD, RB>(P, w, vcur, kspan, kord_s);
                if (it.ntiles == 0) continue;
                const TileInfo my = u == 0 ? it.tu[0] : it.tu[1];
                const bool on = active(it, u);
                auto has = [&](int n) { return it.t0 + n >= my.t0 && it.t0 + n < my.t0 + my.ntiles; };
                auto last_of_u = [&](int n) { return it.t0 + n == my.t0 + my.ntiles - 1; };
                // S(n) = Q_u K(n)^T into S_u; the item's last S also frees the Q slot
                auto issue_s = [&](int n) {
                    const int gs = (g + n) % NS;
                    const uint64_t kdesc = sdesc_sw128(sbase + C::kKOff + gs * C::kKVBytes, 16, 1024);
                    // descriptor + (byte offset >> 4) moves the start address (no carry below 256 KB)
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off_q = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
                        const uint32_t off_k = ((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4;
                        mma_ss_e(tS, qdesc + off_q, kdesc + off_k, idS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_e(BAR(S_FULL(u)));
                    if (last_of_u(n)) mma_commit_e(BAR(Q_EMPTY(u)));
                };
                // O_u (+)= P_u V(n); the item's last one signals the epilogue
                auto issue_pv = [&](int n, int k) {
                    const int vs = (g + n) % NS;
                    const uint64_t vdesc = sdesc_sw128(sbase + C::kVOff + vs * C::kKVBytes, BN * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts_e(tO, tS + kk * 8, vdesc + ((kk * 16 * 128) >> 4), idPV,
                                   (k > 0 || kk > 0) ? 1u : 0u);
                    if (k == my.ntiles - 1) mma_commit_e(BAR(O_DONE(u)));
                };
                // Each step first waits for V(n) and K(n+1) (normally long resident), so
                // that once P(n) arrives PV(n) and S(n+1) issue back to back.  The stage
                // releases count arrivals, not issuers: a chain commits a tile's release
                // only after it has waited for that tile's data phase (also for tiles it
                // skips), so an arrival can never belong to a later use of the stage.
                if (on && !wait_all(ROPE ? Q_ROT(u) : Q_FULL(u), act & 1)) {
                    ok = false;
                    break;
                }
                if (!wait_all(K_FULL(g % NS), (g / NS) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (has(0)) issue_s(0);
                mma_commit_e(BAR(K_EMPTY(g % NS)));
                for (int n = 0; ok && n < it.ntiles; ++n) {
                    const int gn = g + n;
                    ok = wait_all(V_FULL(gn % NS), (gn / NS) & 1);
                    if (ok && n + 1 < it.ntiles) ok = wait_all(K_FULL((gn + 1) % NS), ((gn + 1) / NS) & 1);
                    const int k = it.t0 + n - my.t0;  // index of tile n in u's own sequence
                    if (ok && has(n)) {
                        ok = wait_all(P_FULL(u), pc & 1);
                        ++pc;
                        // the first P.V overwrites O_u: the previous item's epilogue must have read it
                        if (ok && k == 0 && act > 0) ok = wait_all(O_EMPTY(u), (act - 1) & 1);
                    }
                    if (!ok) break;
                    tc_fence_after();
                    if (has(n)) issue_pv(n, k);
                    if (n + 1 < it.ntiles && has(n + 1)) issue_s(n + 1);
                    mma_commit_e(BAR(V_EMPTY(gn % NS)));
                    if (n + 1 < it.ntiles) mma_commit_e(BAR(K_EMPTY((gn + 1) % NS)));
                }
                g += it.ntiles;
                if (on) ++act;
            }
            mma_commit_e(BAR(MMA_DONE));
            mbar_wait(BAR(MMA_DONE), 0, P.status, ST_TEARDOWN, nullptr);
        }  // warp 11 only fills the producer warpgroup
    } else {
        regs_inc<kRegsSoftmax>();
        // -------------------------------------- softmax + epilogue of tile u
        const int u = warp >> 2, wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tbase + u * 128, tO = tbase + 256 + u * HD;
        const float sl2 = P.scale_log2;
        const uint64_t sl2_2 = f2_make(sl2, sl2);
        constexpr bool cap = (MODE & 4) != 0;
        const float cap_in = P.scale / fmaxf(P.softcap, 1e-30f);
        const float cap_out = P.softcap * kLog2e;
        auto wait_warp = [&](int bar, uint32_t parity) -> bool {
            const bool rr = mbar_wait(BAR(bar), parity, P.status, ST_FWD_SOFTMAX, &abort_flag);
            return __all_sync(0xffffffffu, rr);
        };
        bool ok = true;
        int sc = 0;   // S_FULL(u) phases consumed
        int act = 0;  // items in which this tile was active so far (O_DONE phases)
        // One tile's softmax, one thread per row.  The row's 128 scores come out of
        // TMEM into registers in one go (four loads in flight), so P can be written
        // over S chunk by chunk as it is formed.  Pass 1 takes the row max (after the
        // invisible scores are set to -inf, in tiles that some row does not see
        // whole); pass 2 forms P = exp2(x) with x = s*scale*log2(e) - m, or with the
        // capped score softcap*tanh(s*scale/softcap)*log2(e) in place of
        // s*scale*log2(e), pairs of scores through the f32x2 unit together.
        //   The reference m (log2 units, starting at 0) moves only when P would leave
        // [2^-2, 2^8] at the row max: a max above 2^8 (any tile), or a first tile whose
        // max is below 2^-2; then O is rescaled in TMEM first.  For ordinary inputs
        // this never happens.  The softcap takes the fitted tanh polynomial unless a
        // raw score of the warp's rows lies outside its range (mode 2: tanh_accurate),
        // and the shorter one when every raw score lies inside its range (mode 3).
        auto run_tile = [&](auto capc, float& m_used, float& l, int k, bool full, int clo, int chi,
                            const uint32_t(&mbits)[4], uint32_t(&sv)[4][32]) {
            constexpr bool kCap = decltype(capc)::value;
            bool accurate = false, shorter = false;
            if constexpr (kCap) {
                // largest raw |score| of the row, before masking
                float am[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        am[c] = max3f(am[c], fabsf(__uint_as_float(sv[c][e])), fabsf(__uint_as_float(sv[c][e + 1])));
                const float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));
                const CapPoly cp = cap_poly(P.scale, P.softcap);
                accurate = __any_sync(0xffffffffu, !(amax <= cp.r_max)) || (!full && !cp.inf_ok);
                const CapShort cs = cap_short(P.scale, P.softcap);
                shorter = !accurate && __all_sync(0xffffffffu, amax <= cs.r_max) && (full || cs.inf_ok);
            }
            if (!full) {
                // visibility bits of columns 32c .. 32c+31: [clo, chi) and the key mask
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int lo = min(max(clo - 32 * c, 0), 32), hi = min(max(chi - 32 * c, 0), 32);
                    const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
                    const uint32_t below_lo = lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u);
                    const uint32_t vw = below_hi & ~below_lo & mbits[c];
#pragma unroll
                    for (int e = 0; e < 32; ++e) sv[c][e] = ((vw >> e) & 1u) ? sv[c][e] : 0xff800000u;  // -inf
                }
            }
            // pass 1: the row max of the scores, as x against the current reference
            float rm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    rm[c] = max3f(rm[c], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
            const float rmax = fmaxf(fmaxf(rm[0], rm[1]), fmaxf(rm[2], rm[3]));
            // x is increasing in the score, so its row max is x(rmax)
            auto to_x = [&](auto modec, uint64_t rr, uint64_t nms) -> uint64_t {
                constexpr int kMode = decltype(modec)::value;
                if constexpr (kMode == 2) {
                    float r0, r1;
                    f2_split(rr, r0, r1);
                    float m0, m1;
                    f2_split(nms, m0, m1);
                    // a masked score is -inf, and softcap*tanh(-inf) would be finite
                    return f2_make(r0 == -INFINITY ? -INFINITY : fmaf(cap_out, tanh_accurate(r0 * cap_in), m0),
                                   r1 == -INFINITY ? -INFINITY : fmaf(cap_out, tanh_accurate(r1 * cap_in), m1));
                } else if constexpr (kMode == 1) {
                    // x = r * (sl2 + u * S'(u)) + m with u = r^2 and S' the fit's S with
                    // scale * log2(e) folded in: one packed operation fewer than g * sl2 + m
                    const CapPoly cp = cap_poly(P.scale, P.softcap);
                    const uint64_t u = f2_mul(rr, rr);
                    uint64_t sp = f2_fma(u, f2_mul(cp.s3, sl2_2), f2_mul(cp.s2, sl2_2));
                    sp = f2_fma(u, sp, f2_mul(cp.s1, sl2_2));
                    sp = f2_fma(u, sp, f2_mul(cp.s0, sl2_2));
                    return f2_fma(rr, f2_fma(u, sp, sl2_2), nms);
                } else if constexpr (kMode == 3) {
                    // the same with the short fit
                    const CapShort cs = cap_short(P.scale, P.softcap);
                    const uint64_t u = f2_mul(rr, rr);
                    const uint64_t sp = f2_fma(u, f2_mul(cs.s1, sl2_2), f2_mul(cs.s0, sl2_2));
                    return f2_fma(rr, f2_fma(u, sp, sl2_2), nms);
                } else {
                    return f2_fma(rr, sl2_2, nms);
                }
            };
            float xm, xm_;
            {
                const uint64_t r2 = f2_make(rmax, rmax), n2 = f2_make(-m_used, -m_used);
                uint64_t x2;
                if (!kCap) x2 = to_x(std::integral_constant<int, 0>(), r2, n2);
                else if (shorter) x2 = to_x(std::integral_constant<int, 3>(), r2, n2);
                else if (!accurate) x2 = to_x(std::integral_constant<int, 1>(), r2, n2);
                else x2 = to_x(std::integral_constant<int, 2>(), r2, n2);
                f2_split(x2, xm, xm_);
            }
            if (rmax == -INFINITY) xm = -INFINITY;
            const bool resc = xm > kRescaleHi || (l == 0.f && xm < kRescaleLo && xm != -INFINITY);
            if (__any_sync(0xffffffffu, resc)) {
                // S_u(k) completed after P_u(k-1) V(k-1): O_u holds every earlier tile.
                // Rows that have seen nothing yet hold O = 0 and keep alpha = 1 (their
                // reference may move down by any amount).
                const float alpha = fast_exp2(resc && l > 0.f ? -xm : 0.f);
                if (resc) {
                    m_used += xm;
                    l *= alpha;
                }
                if (k > 0) {
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
            // pass 2: P chunk by chunk, each 16-bit chunk stored over S as soon as formed
            auto p_pass = [&](auto modec) {
                const uint64_t nms = f2_make(-m_used, -m_used);
                uint64_t rs2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0, x1;
                        f2_split(to_x(modec, f2_make(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])), nms),
                                 x0, x1);
                        const float p0 = fast_exp2(x0);  // ex2(-inf) = 0
                        const float p1 = fast_exp2(x1);
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
            if (!kCap) p_pass(std::integral_constant<int, 0>());
            else if (shorter) p_pass(std::integral_constant<int, 3>());
            else if (!accurate) p_pass(std::integral_constant<int, 1>());
            else p_pass(std::integral_constant<int, 2>());
        };
        // The two tiles' softmaxes alternate A(k), B(k), A(k+1), ... within an item, so
        // each runs while the tensor core works on the other tile's P.V and next S; left
        // alone they fall into lockstep and the tensor core idles during both.  (With a
        // softcap, both at once measured faster while each MMA issue took a branch
        // around it; with the predicated issue the turns win there too, except with a
        // bias as well, whose longer softmax still runs better with both at once.)
        // base[u] counts tile u's softmaxes in earlier items.
        constexpr bool kTurns = !(BIAS && cap);
        int base[2] = {0, 0};
        // Fused rotary embedding: turn this thread's row of tile u's Q in shared memory
        // once the tile of item w2 has landed, then release it to the MMA warp.  Pairs
        // (c, c + hd/2) sit in the same 16-byte chunk slot of the two 64-column boxes
        // (hd 128) or four chunks apart in the one box (hd 64).
        int qr = 0;        // Q tiles of this tile slot rotated so far
        int rot_kw = -1;   // position (in this CTA's item sequence) of the last rotated item
        auto rotate_q = [&](int kw2) -> bool {
            const FwdItem it2 = fwd_item<VL, KORD, RB>(P, snake_item(kw2), vcur, kspan, kord_s);
            const TileInfo my2 = u == 0 ? it2.tu[0] : it2.tu[1];
            if (it2.ntiles == 0 || my2.ntiles == 0) return true;  // the tile is not loaded for this item
            if (!wait_warp(Q_FULL(u), qr & 1)) return false;
            ++qr;
            const int i2 = it2.i0 + u * BM + r;
            if (i2 < it2.sq.tq) {
                // cosine and sine of pair c at this row's position: tab2[c * npos + s]
                const float2* tcol = reinterpret_cast<const float2*>(P.rope_tab) + (P.q_offset + i2);
                uint8_t* qrow = smem + C::kQOff + u * C::kQBytes + r * 128;
#pragma unroll
                for (int j = 0; j < HD / 16; ++j) {
                    uint4* pa = reinterpret_cast<uint4*>(qrow + ((j ^ (r & 7)) << 4));
                    uint4* pb = reinterpret_cast<uint4*>(HD == 128 ? qrow + BM * 128 + ((j ^ (r & 7)) << 4)
                                                                   : qrow + (((j + 4) ^ (r & 7)) << 4));
                    uint4 a = *pa, b = *pb;
                    uint32_t* aw = reinterpret_cast<uint32_t*>(&a);
                    uint32_t* bw = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 c0 = __ldg(tcol + (long long)(8 * j + 2 * e) * P.rope_npos);
                        const float2 c1 = __ldg(tcol + (long long)(8 * j + 2 * e + 1) * P.rope_npos);
                        const float4 cs = make_float4(c0.x, c0.y, c1.x, c1.y);  // pairs 8j+2e and 8j+2e+1
                        float a0, a1, b0, b1, ra0, ra1, rb0, rb1;
                        if constexpr (BF16) {
                            const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
                            const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[e]));
                            a0 = fa.x; a1 = fa.y; b0 = fb.x; b1 = fb.y;
                        } else {
                            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&aw[e]));
                            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&bw[e]));
                            a0 = fa.x; a1 = fa.y; b0 = fb.x; b1 = fb.y;
                        }
                        rope_turn(a0, b0, cs.x, cs.y, ra0, rb0);
                        rope_turn(a1, b1, cs.z, cs.w, ra1, rb1);
                        aw[e] = pack2<BF16>(ra0, ra1);
                        bw[e] = pack2<BF16>(rb0, rb1);
                    }
                    *pa = a;
                    *pb = b;
                }
            }
            fence_proxy_async_smem();  // the tensor core reads the tile through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_ROT(u)));
            rot_kw = kw2;
            return true;
        };
        for (int kw = 0, w = snake_item(0); ok && w < nitems; w = snake_item(++kw)) {
            const FwdItem it = fwd_item<VL, KORD, RB>(P, w, vcur, kspan, kord_s);
            const int nA = it.tu[0].ntiles, nB = it.tu[1].ntiles;
            const int bA = base[0], bB = base[1];
            // The turns pair the tiles' k-th key tiles.  A tile whose first key tile lies
            // more than one behind the other's could wait for a turn whose S needs a K/V
            // ring stage that only its own later P.V releases (packed fused-QKV rows,
            // where a tile that ends a long sequence starts many key tiles before the
            // next one): such items run both softmaxes at once.
            const bool alt = kTurns && abs(it.tu[0].t0 - it.tu[1].t0) <= 1;
            base[0] += nA;
            base[1] += nB;
            const int ib = it.i0 + u * BM;  // first row of this tile
            if (ib >= it.sq.tq) continue;
            const int tq = it.sq.tq, tk = it.sq.tk;
            const int i = ib + r;
            const int p = i + P.q_offset;
            const int prow0 = ib + P.q_offset, prow1 = min(ib + BM, tq) - 1 + P.q_offset;
            const TileInfo my = u == 0 ? it.tu[0] : it.tu[1];
            // packed fused-QKV rows: this row's sequence, and the keys every row of the tile sees
            int2 rk_own = make_int2(0, tk), rk_all = make_int2(0, tk);
            if constexpr (RB) {
                rk_own = row_keys(P, max(min(i, tq - 1), 0), tk);
                rk_all = make_int2(row_keys(P, min(ib + BM, tq) - 1, tk).x, row_keys(P, ib, tk).y);
            }
            if constexpr (ROPE) {
                // this item's Q, unless the previous item's end already turned it
                if (my.ntiles > 0 && rot_kw != kw && !rotate_q(kw)) {
                    ok = false;
                    break;
                }
            }
            float m_used = 0.f, l = 0.f;
            for (int k = 0; k < my.ntiles; ++k) {
                const int j0 = (my.t0 + k) * BN;
                uint32_t mbits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
                if (P.key_mask) {
                    const float* mrow = P.key_mask + (long long)it.b * P.mask_bstride;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int j = j0 + c * 32 + lane;
                        mbits[c] = __ballot_sync(0xffffffffu, j < tk && mrow[j] > 0.5f);
                    }
                }
                // a tile whose keys the mask keeps whole needs no mask pass
                const bool full = tile_full(P.wl, P.wr, tk, prow0, prow1, j0, j0 + BN) &&
                                  (mbits[0] & mbits[1] & mbits[2] & mbits[3]) == 0xffffffffu &&
                                  (!RB || (j0 >= rk_all.x && j0 + BN <= rk_all.y));
                // this row's visible columns of the tile: [clo, chi), and the key-mask bits
                int clo = 0, chi = BN;
                if (!full) {
                    chi = min(chi, tk - j0);
                    if (P.wr >= 0) chi = min(chi, p + P.wr - j0 + 1);
                    if (P.wl >= 0) clo = max(clo, p - P.wl - j0);
                    if constexpr (RB) {
                        clo = max(clo, rk_own.x - j0);
                        chi = min(chi, rk_own.y - j0);
                    }
                }
                // additive score bias: loads issued before the waits
                float bv[BIAS ? 128 : 1];
                if constexpr (BIAS) {
                    if (i < tq) load_bias_row(P, it.b, it.h, i, j0, tk, bv);
                    else
#pragma unroll
                        for (int e = 0; e < 128; ++e) bv[e] = 0.f;
                }
                if (!wait_warp(S_FULL(u), sc & 1)) {
                    ok = false;
                    break;
                }
                ++sc;
                tc_fence_after();
                // the row's 128 scores, loaded while this tile waits for its turn (with a
                // bias, a chunk at a time after the wait, each gaining its bias as it lands)
                uint32_t sv[4][32];
                if constexpr (!BIAS) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, sv[c]);
                }
                if (alt && (u == 0 ? (k >= 1 && k - 1 < nB) : (k < nA))) {
                    const int need = 4 * (u == 0 ? bB + k : bA + k + 1);  // warp arrivals
                    const bool rr = count_wait(&done_count[u ^ 1], need, P.status, ST_FWD_SOFTMAX, &abort_flag);
                    if (!__all_sync(0xffffffffu, rr)) {
                        if constexpr (!BIAS) tmem_ld_wait_only();
                        ok = false;
                        break;
                    }
                }
                if constexpr (BIAS) {
                    const float inv = 1.f / P.scale;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld32(tS + lane_off + c * 32, sv[c]);
                        tmem_ld_wait(sv[c]);
                        if constexpr (cap) {
                            // the cap comes before the bias: the capped score in raw-score
                            // units, g = tanh(s * scale / softcap) * softcap / scale, by the
                            // fitted polynomial where every raw score of the warp's chunk lies
                            // in its range, else by the exp-based tanh
                            const CapPoly cp = cap_poly(P.scale, P.softcap);
                            float am = 0.f;
#pragma unroll
                            for (int e = 0; e < 32; e += 2)
                                am = max3f(am, fabsf(__uint_as_float(sv[c][e])), fabsf(__uint_as_float(sv[c][e + 1])));
                            if (__all_sync(0xffffffffu, am <= cp.r_max)) {
#pragma unroll
                                for (int e = 0; e < 32; e += 2) {
                                    uint64_t uu;
                                    float g0, g1;
                                    f2_split(cap_g(cp, f2_make(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), uu),
                                             g0, g1);
                                    sv[c][e] = __float_as_uint(g0);
                                    sv[c][e + 1] = __float_as_uint(g1);
                                }
                            } else {
                                const float cap_in = P.scale / P.softcap, cap_back = P.softcap / P.scale;
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    sv[c][e] = __float_as_uint(tanh_accurate(__uint_as_float(sv[c][e]) * cap_in) * cap_back);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            sv[c][e] = __float_as_uint(fmaf(bv[32 * c + e], inv, __uint_as_float(sv[c][e])));
                    }
                } else {
                    tmem_ld_wait_only();
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_pin(sv[c]);
                }
                // (with a bias the cap was applied above, before the bias)
                if (cap && !BIAS) run_tile(std::integral_constant<bool, true>(), m_used, l, k, full, clo, chi, mbits, sv);
                else run_tile(std::integral_constant<bool, false>(), m_used, l, k, full, clo, chi, mbits, sv);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(BAR(P_FULL(u)));
                    atomicAdd(&done_count[u], 1);
                }
            }
            if constexpr (ROPE) {
                // the next item's Q lands once this item's last S of the tile completed:
                // turn it now, so that its first S need not wait for this epilogue
                if (ok && snake_item(kw + 1) < nitems && !rotate_q(kw + 1)) ok = false;
            }
            const bool have_o = ok && my.ntiles > 0 && wait_warp(O_DONE(u), act & 1);
            if (my.ntiles > 0) ++act;
            if (have_o) tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint32_t packed[HD / 2];
            {
                // all of the row's O columns in flight at once, one wait
                uint32_t orr[HD / 32][32];
                if (have_o) {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) tmem_ld32(tO + lane_off + c * 32, orr[c]);
                    tmem_ld_wait_only();
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) tmem_pin(orr[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[c][e] = 0u;
                }
#pragma unroll
                for (int c = 0; c < HD / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        packed[c * 16 + e] = pack2<BF16>(__uint_as_float(orr[c][2 * e]) * inv,
                                                         __uint_as_float(orr[c][2 * e + 1]) * inv);
            }
            // O_u is in registers: the next item's first P.V may overwrite it
            if (have_o) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(O_EMPTY(u)));
            }
            // A packed sequence's last rows may share a 32-row slice with the next
            // sequence's first: such a slice goes out row by row (rows of this sequence
            // only).  Dense tensors end where the map ends, which clips the tiled store.
            const bool whole = !VL || ib + wq * 32 + 32 <= tq;
            if (ok && (have_o || my.ntiles == 0) && !whole && i < tq) {
                uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(P.o) +
                                                       ((long long)it.sq.q0 + i) * P.H * HD + (long long)it.h * HD);
#pragma unroll
                for (int w4 = 0; w4 < HD / 8; ++w4)
                    orow[w4] = make_uint4(packed[4 * w4], packed[4 * w4 + 1], packed[4 * w4 + 2], packed[4 * w4 + 3]);
            }
            if (ok && (have_o || my.ntiles == 0) && whole) {
                // This warp's 32 rows go out through its 4 KB staging slice, 64 columns
                // at a time, in the 128-byte-swizzled layout of the tensor map's box;
                // one lane issues the tiled store (rows past Tq are not written).
                const uint32_t slice = sbase + C::kStgOff + (u * 4 + wq) * 4096;
#pragma unroll
                for (int half = 0; half < HD / 64; ++half) {
                    if (elect_one()) bulk_wait_read_all();  // the slice's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int w4 = half * 32 + 4 * j;
                        st_shared_v4(slice + lane * 128 + ((j ^ (lane & 7)) << 4), packed[w4], packed[w4 + 1],
                                     packed[w4 + 2], packed[w4 + 3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (elect_one()) {
                        tile_store<PADH, HD>(&tmO, slice, it.h, half * 64, it.sq.q0 + ib + wq * 32, it.sq.zb);
                        bulk_commit_group();
                    }
                }
            }
            if (ok && (have_o || my.ntiles == 0) && P.lse && i < tq)
                P.lse[((long long)it.b * P.H + it.h) * P.Tq + i] =
                    l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
            if (!ok) break;
        }
        // the staging slice must stay until this warp's last store has read it
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

template <bool BF16, int HD>
cudaError_t fwd2_typed(const Params& p, const FwdMaps& m, cudaStream_t s) {
    using C = Fwd2Cfg<HD>;
    const bool c = p.softcap > 0.f;
    // a head size below HD (dense batches without a bias only) runs the padded instantiations
    // the rotary query turn (dense batches at hd 64 / 128) runs the MODE & 16 instantiations
    // packed fused-QKV rows (one dense batch at hd 64 / 128, no other mode) run MODE 64
    auto kern = p.rope_tab  ? (c ? fwd_tc2_kernel<BF16, HD, 20> : fwd_tc2_kernel<BF16, HD, 16>)
                : p.row_bounds ? fwd_tc2_kernel<BF16, HD, 64>
                : p.hd != HD ? (c ? fwd_tc2_kernel<BF16, HD, 12> : fwd_tc2_kernel<BF16, HD, 8>)
                : p.cu_q   ? (c ? fwd_tc2_kernel<BF16, HD, 5> : fwd_tc2_kernel<BF16, HD, 1>)
                : p.bias   ? (c ? fwd_tc2_kernel<BF16, HD, 6> : fwd_tc2_kernel<BF16, HD, 2>)
                : c        ? fwd_tc2_kernel<BF16, HD, 4>
                : p.key_mask && p.B <= kMaskSpanMax ? fwd_tc2_kernel<BF16, HD, 32>
                                                    : fwd_tc2_kernel<BF16, HD, 0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kLaunchBytes);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // persistent: one CTA per SM (one fits), each walks its items in snake order
    // (packed sequences may have fewer items than this bound: those CTAs exit at once)
    const long long items = (long long)((p.Tq + 2 * BM - 1) / (2 * BM)) * p.H * p.B;
    const unsigned grid = (unsigned)(items < nsm ? items : nsm);
    kern<<<grid, kThreads2, C::kLaunchBytes, s>>>(p, m.q, m.k, m.v, m.o);
    return cudaGetLastError();
}

}  // namespace

}  // namespace attn
